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

// Threads per CTA of the ring and lock-step kernels: 16 warps while the
// R x M partial sums and the unpacked weights fit in 128 registers (the
// top-1 forms at M = 4 and 6 included: 112 and 127 registers, and 16 warps
// made the six-row fused head 6 us faster than the unfused path, where 12
// had left it level); 12 warps (168 registers) for M = 7 .. 16, and for the
// top-k form at M = 3 and 4, which would spill with 16 (12 warps took the
// Q6_K heads at M = 9, 12 and 16 from 294 / 356 / 446 to 280 / 351 / 441 us
// against 8; 16 instead of 12 took the top-8 at M = 5 from 225 to 214 us);
// 8 warps (255 registers) for M = 17.
template <int FMT, int M, bool TOP1, bool TOPK = false>
struct MmvqThreads {
    static constexpr bool wide = M == 7 || M == 8 || (TOPK && (M == 3 || M == 4));
    static constexpr int value = M > 16 ? 256 : (M > 8 || wide ? 384 : 512);
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

// Q6_K: the code bytes P and Q, the subscales of the block for row r, dw[r] =
// its superblock scale.
template <int M, int R>
__device__ __forceinline__ void accumulate_q6_k(const uint4 (&cp)[R], const uint2 (&cq)[R], const uint32_t (&sc)[R],
                                                const float (&dw)[R], const ActTile& t, int ti, float (&acc)[R][M])
{
    uint32_t w[R][8];
    float dq[R];  // the superblock scale over four (q6_k_dot returns 4 J)
#pragma unroll
    for (int r = 0; r < R; ++r) {
        q6_k_unpack(cp[r], cq[r], w[r]);
        dq[r] = dw[r] * 0.25f;
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 lo = t.aq[(m * 2 + 0) * t.KC + ti];
        const uint4 hi = t.aq[(m * 2 + 1) * t.KC + ti];
        const uint2 mt = t.am[m * t.KC + ti];
        const float da = __uint_as_float(mt.x);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int J4 = q6_k_dot(w[r], lo, hi, mt.y, sc[r]);
            acc[r][m] = fmaf(dq[r] * da, (float)J4, acc[r][m]);
        }
    }
}

// ---------------------------------------------------------------------------
// Activation tile of the ring kernel, block-major: block b's codes for rows
// m = 0..M-1 lie at q + b * QSTRIDE + 32 m (two 16-byte halves); QSTRIDE is an
// odd number of 16-byte units, so the 32 lanes of a warp, which read 32
// consecutive blocks, touch 32 distinct 16-byte bank groups (4 wavefronts,
// no conflict).  Block b's per-row words lie at meta + (b * MROWS + m) * META
// with MROWS = M rounded up to odd, for the same reason:
//   Q4_0 (8 B):  fp32 bits of the fp16 scale d_a;  -8 * sum(q) + 0x4B400000
//   Q6_K (16 B): fp32 bits of d_a; -32 * sum(q[0..15]); -128 * sum(q[16..31]); 0
// The integer words start the dp4a chains, folding the weight offsets
// (q_w - 8, q_w - 32) in exactly (the Q6_K second half's codes come four
// times over, q6_k_unpack); the Q4_0 one also carries the bias of the
// int -> float conversion below.
// ---------------------------------------------------------------------------

template <int FMT, int M>
struct RingAct {
    static constexpr int QSTRIDE = (2 * M + 1) * 16;
    static constexpr int MROWS = M | 1;
    static constexpr int META = FMT == FMT_Q4_0 ? 8 : 16;
    __host__ __device__ static constexpr size_t bytes(int NB)
    {
        return (size_t)NB * (size_t)(QSTRIDE + MROWS * META);
    }
    uint8_t* q;
    uint8_t* meta;
};

template <int FMT>
__device__ __forceinline__ void ring_meta_store(uint8_t* p, float da, int s_lo, int s_hi)
{
    if (FMT == FMT_Q4_0) {
        *reinterpret_cast<uint2*>(p) =
            make_uint2(__float_as_uint(da), (uint32_t)(-8 * (s_lo + s_hi) + MAGIC_I2F_BITS));
    } else {
        // the second half's codes come four times over (q6_k_unpack)
        *reinterpret_cast<uint4*>(p) = make_uint4(__float_as_uint(da), (uint32_t)(-32 * s_lo), (uint32_t)(-128 * s_hi), 0u);
    }
}

// From caller-supplied Q8_1 blocks in global memory: each thread takes U
// blocks per round and issues all their loads before using any, so a round
// costs one L2 round trip.  U = 4 for the short Q4_0 calls, whose staging is
// a visible part of the call (the down projection stages 3264 blocks); the
// Q6_K heads keep U = 1, which leaves their main loop's registers alone.
template <int FMT, int M>
__device__ __forceinline__ void ring_act_from_q8_1(const RingAct<FMT, M>& t, const uint8_t* xq, int NB)
{
    using A = RingAct<FMT, M>;
    constexpr int U = FMT == FMT_Q4_0 ? 4 : 1;
    const int total = M * NB;
    for (int i0 = threadIdx.x; i0 < total; i0 += U * blockDim.x) {
        uint32_t w[U][9];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * blockDim.x;
            if (i < total) {
                const uint32_t* src = reinterpret_cast<const uint32_t*>(xq + (int64_t)i * Q8_1_BYTES);
#pragma unroll
                for (int k = 0; k < 9; ++k) w[u][k] = src[k];
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * blockDim.x;
            if (i >= total) break;
            const int m = i / NB, b = i - m * NB;
            uint4* dst = reinterpret_cast<uint4*>(t.q + b * A::QSTRIDE + 32 * m);
            dst[0] = make_uint4(w[u][1], w[u][2], w[u][3], w[u][4]);
            dst[1] = make_uint4(w[u][5], w[u][6], w[u][7], w[u][8]);
            int s0 = 0, s1 = 0;
#pragma unroll
            for (int k = 1; k < 5; ++k) s0 = __dp4a((int)w[u][k], 0x01010101, s0);
#pragma unroll
            for (int k = 5; k < 9; ++k) s1 = __dp4a((int)w[u][k], 0x01010101, s1);
            const float da = __half2float(__ushort_as_half((unsigned short)(w[u][0] & 0xFFFFu)));
            ring_meta_store<FMT>(t.meta + (b * A::MROWS + m) * A::META, da, s0, s1);
        }
    }
}

// From fp32 activations, quantizing to Q8_1 on the fly with 8 lanes per block
// (four blocks per warp step), bit-identical to the quantize_q8_1 kernel.
template <int FMT, int M>
__device__ __forceinline__ void ring_act_from_f32(const RingAct<FMT, M>& t, const float* x, int64_t ldx, int NB)
{
    using A = RingAct<FMT, M>;
    const bool vec4 = ((reinterpret_cast<uintptr_t>(x) | ((uintptr_t)ldx * 4)) & 15u) == 0;
    const int lane = threadIdx.x & 31, sub = lane & 7, W = blockDim.x >> 5;
    const int nblk = M * NB;
    for (int i0 = (threadIdx.x >> 5) * 4; i0 < nblk; i0 += W * 4) {  // warp-uniform
        const int mine = i0 + (lane >> 3);
        const int i = mine < nblk ? mine : nblk - 1;  // spare lanes redo the last block, unwritten
        const int m = i / NB, b = i - m * NB;
        const Q81Lanes o = q8_1_quantize_8lanes(load_4_values(x + (int64_t)m * ldx + b * QK + 4 * sub, vec4));
        if (mine < nblk) {
            *reinterpret_cast<uint32_t*>(t.q + b * A::QSTRIDE + 32 * m + 4 * sub) = o.word;
            if (sub == 0)
                ring_meta_store<FMT>(t.meta + (b * A::MROWS + m) * A::META, __half2float(__float2half_rn(o.d)),
                                     o.s_half, o.s_all - o.s_half);
        }
    }
}

// ---------------------------------------------------------------------------
// Kernel arguments and epilogue.
// ---------------------------------------------------------------------------

struct MmvqArgs {
    const void* w_pack;
    const uint8_t* xq;  // Q8_1 [M][NB]; null (top-1 kernels only): quantize x in the kernel
    const float* x;     // fp32 [M][ldx] (when xq is null); the residual of a RES kernel
    int64_t ldx;
    union {
        struct {
            float* y;  // the output [M][ldy] (kernels that write one)
            int64_t ldy;
        };
        struct {
            // top-k kernels (which write no output): each CTA's k best keys
            // per row, [grid][M][k], merged by the last CTA; and k
            unsigned long long* topk_lists;
            int64_t topk;
        };
    };
    int K, N;
    // optional second weight of the same K against the same activation (a
    // pair such as gate and up): its row groups follow the first's
    const void* w_pack2;
    float* y2;
    int N2;
    int KC;      // activation blocks staged at once (lock-step kernel)
    int stages;  // ring stages per warp (ring kernel)
    int parts;   // K parts per row group (ring kernel)
    Top1Workspace* ws;
    int32_t* ids;
    // candidate-max (top-1 kernels, all optional): the top value of each row,
    // and the logit of a given candidate id per row
    float* top_vals;  // (top-k kernels: [M][k], as ids)
    const int32_t* cand;
    float* cand_vals;
#ifdef QGEMV_BOUNDS_CHECK
    // test hook: move the first stores of CTA 0, warp 0 out of their extent,
    // for the bounds check to catch
    int plant_bad_store;
#endif
};

// Debug-build checks of the ring and lock-step kernels' computed accesses.
// A weight copy must lie in the pack of the first weight or, for a pair, of
// the second; an output (m, n) in the [M][ldy] output of its weight.
__device__ __forceinline__ bool pack_range_ok(const MmvqArgs& a, int fmt, const uint8_t* src, uint32_t bytes)
{
    const int64_t o0 = (int64_t)(reinterpret_cast<uintptr_t>(src) - reinterpret_cast<uintptr_t>(a.w_pack));
    if (qg_in(o0, bytes, make_layout(fmt, a.N, a.K).total_bytes())) return true;
    if (!a.w_pack2) return false;
    const int64_t o1 = (int64_t)(reinterpret_cast<uintptr_t>(src) - reinterpret_cast<uintptr_t>(a.w_pack2));
    return qg_in(o1, bytes, make_layout(fmt, a.N2, a.K).total_bytes());
}

__device__ __forceinline__ bool store_ok(const MmvqArgs& a, const float* y, int m, int M, int64_t n)
{
    const int Ny = (a.y2 && y == a.y2) ? a.N2 : a.N;
    return m >= 0 && m < M && n >= 0 && n < Ny;
}

// Bytes of dynamic shared memory the kernel was launched with.
__device__ __forceinline__ uint32_t dynamic_smem_bytes()
{
    uint32_t v;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(v));
    return v;
}

// Output store of a plain MMVQ; the residual instantiation (RES) adds the
// residual, which such calls pass in the fp32-activation field x (row stride
// ldx), as each output is stored (the same thread reads and writes the
// element, so the residual may be y itself).
template <bool RES>
__device__ __forceinline__ void mmvq_store(const MmvqArgs& a, float* y, int m, int64_t n, float v)
{
    y[(int64_t)m * a.ldy + n] = RES ? v + a.x[(int64_t)m * a.ldx + n] : v;
}

// Reduce one row group's partial sums over the warp and write them (TOP1 =
// false) or fold their keys into the warp's running best per row (TOP1).
template <int M, int R, bool TOP1, bool RES = false>
__device__ __forceinline__ void finish_rowgroup(const MmvqArgs& a, int n0, float (&acc)[R][M], int lane,
                                                unsigned long long* wk, unsigned long long& best, unsigned int* status)
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
                    if (n < a.N && QG_OK(store_ok(a, a.y, m, M, n), status, 720))
                        mmvq_store<RES>(a, a.y, m, n, v[j]);
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
                    if (a.cand_vals && n < a.N && n == a.cand[vi % M]) a.cand_vals[vi % M] = v[j];
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
            if (a.top_vals) a.top_vals[threadIdx.x] = top1_key_to_value(k);
        }
        if (threadIdx.x == 0) atomicExch(&a.ws->done, 0u);
    }
}

// ---------------------------------------------------------------------------
// Top-k on the same ordered keys.  Keys are unique (the id is part of the
// key), so the k largest keys of a row form one set whatever the order in
// which they are kept, merged or selected: the result is deterministic.
// 0 is "no key" (a NaN, or no entry), below every real key.  Each warp keeps
// one list per row, each CTA merges its warps' lists, and the last CTA
// merges the CTAs' lists.
// ---------------------------------------------------------------------------

constexpr int TOPK_MAX = 8;

// Whole warp.  Each lane offers NR keys (0: none), key j for row row[j], to
// the warp's lists wl[row * TOPK_MAX + i], i < k, kept in descending order
// (0-filled).  A key enters only if it beats the row's k-th key; such keys
// are taken one at a time, the k lanes of the list shifting it down by one.
template <int NR>
__device__ __forceinline__ void topk_offer(unsigned long long* wl, int k, const unsigned long long (&key)[NR],
                                           const int (&row)[NR], int lane)
{
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        unsigned int mask = __ballot_sync(0xffffffffu, key[j] > wl[row[j] * TOPK_MAX + k - 1]);
        while (mask) {
            const int src = __ffs(mask) - 1;
            mask &= mask - 1;
            const unsigned long long kk = __shfl_sync(0xffffffffu, key[j], src);
            unsigned long long* list = wl + __shfl_sync(0xffffffffu, row[j], src) * TOPK_MAX;
            const unsigned long long cur = lane < k ? list[lane] : 0ull;
            // entries that stay above it (the threshold may have risen since
            // the ballot: then pos == k and nothing moves)
            const int pos = __popc(__ballot_sync(0xffffffffu, lane < k && cur > kk));
            const unsigned long long up = __shfl_up_sync(0xffffffffu, cur, 1);
            if (lane < k && lane >= pos) list[lane] = lane == pos ? kk : up;
            __syncwarp();
        }
    }
}

// Whole warp: the k largest of `count` keys load(e), e < count, handed to
// out(r, key) by lane 0 in descending order (r = 0..k-1); when fewer than k
// keys are nonzero the remaining picks are 0.  k rounds, each a strided scan
// for the largest key below the previous pick and a warp maximum.
template <class Load, class Out>
__device__ __forceinline__ void topk_select(int count, int k, int lane, Load load, Out out)
{
    unsigned long long prev = ~0ull;
    for (int r = 0; r < k; ++r) {
        unsigned long long best = 0ull;
        for (int e = lane; e < count; e += 32) {
            const unsigned long long x = load(e);
            if (x < prev && x > best) best = x;
        }
        best = warp_max_u64(best);
        if (lane == 0) out(r, best);
        prev = best;
    }
}

// Whole warp: the k largest keys of `n` lists, each sorted larger first and
// 0-filled, list j at lists[j * stride .. + k - 1], handed to out(r, key) by
// lane 0 in descending order (0 once the lists hold no more keys).  Lane l
// holds the heads of lists l, l + 32, ... (n <= 32 * TOPK_HEADS); each round
// is a warp maximum over the heads, and the list holding the winner (keys are
// unique) moves its head on.
constexpr int TOPK_HEADS = 8;
template <class Out>
__device__ __forceinline__ void topk_merge_sorted(const unsigned long long* lists, int n, int stride, int k, int lane,
                                                  Out out)
{
    int head[TOPK_HEADS];
#pragma unroll
    for (int j = 0; j < TOPK_HEADS; ++j) head[j] = 0;
    for (int r = 0; r < k; ++r) {
        unsigned long long best = 0ull;
#pragma unroll
        for (int j = 0; j < TOPK_HEADS; ++j) {
            const int c = lane + 32 * j;
            if (c < n && head[j] < k) {
                const unsigned long long x = lists[(size_t)c * stride + head[j]];
                best = x > best ? x : best;
            }
        }
        best = warp_max_u64(best);
        if (lane == 0) out(r, best);
        if (best == 0ull) continue;
#pragma unroll
        for (int j = 0; j < TOPK_HEADS; ++j) {
            const int c = lane + 32 * j;
            if (c < n && head[j] < k && lists[(size_t)c * stride + head[j]] == best) ++head[j];
        }
    }
}

// Keys a warp folds per row group in the lock-step top-1 kernel: R rows x M
// activation rows, at most R_ROWS * MAX_M.
constexpr int TOP1_GROUP_KEYS = R_ROWS * MAX_M;

// Shared memory besides the activation tile and the rings, for TOP1.
inline size_t top1_scratch_bytes(int nwarps)
{
    return (size_t)nwarps * TOP1_GROUP_KEYS * 8 + (size_t)nwarps * MAX_M * 8 + 16;
}

// ---------------------------------------------------------------------------
// Ring kernel: the whole activation in shared memory, the weights streamed
// through a private ring of S stages per warp, filled by TMA bulk copies.
//   shared memory: row space | copy streams [W] | rings [W][S][CB] | tile codes |
//                  tile meta | mbarriers [W][S] | partial sums [groups][P][4 M]
//                  (P > 1) | top-1 keys
// The CTA owns row groups g0 .. g1-1 (4 rows each).  Each group's K is cut
// into the same P parts (chunks p nch / P .. (p + 1) nch / P - 1), so a group
// is P items; warp w takes items w, w + W, ...  A job is one chunk of an item: one bulk copy of
// the group-chunk (CB bytes) into the warp's next stage, completing on the
// stage's mbarrier; lane 0 issues it S - 1 jobs ahead.  Lane l works on block
// l of the chunk for the four rows, so one activation block feeds four rows
// and one weight block M rows.  With P > 1 the parts' sums meet in shared
// memory and are added in part order, so every output is summed the same way
// wherever its row sits.  Waits are bounded: a warp that waits about a second
// for a copy counts a timeout in *timeouts, stops, and gives its copies in
// flight a bounded wait.
// ---------------------------------------------------------------------------

// Warp reduction of a row group's V = R * M sums, 32 at a time: chunk k
// (sums 32 k .. 32 k + 31, the last one shorter) is transpose-reduced, and
// lane `lane` keeps the total of value ring_value_index<V>(k, lane).
template <int V>
__device__ __forceinline__ int ring_value_index(int k, int lane)
{
    constexpr int LAST = 32 * ((V - 1) / 32);
    constexpr int PL = next_pow2(V - LAST);
    return 32 * k + (32 * k == LAST ? reduced_value_index<PL>(lane, 0) : lane);
}

template <int V>
__device__ __forceinline__ bool ring_value_owner(int k, int lane)
{
    constexpr int LAST = 32 * ((V - 1) / 32);
    constexpr int PL = next_pow2(V - LAST);
    return 32 * k != LAST || (reduced_value_owner<PL>(lane) && reduced_value_index<PL>(lane, 0) < V - LAST);
}

template <int M, int R>
__device__ __forceinline__ void ring_reduce(const float (&acc)[R][M], float (&out)[(R * M + 31) / 32], int lane)
{
    constexpr int V = R * M;
    constexpr int NRED = (V + 31) / 32;
    constexpr int LAST = 32 * (NRED - 1);
    constexpr int PL = next_pow2(V - LAST);
#pragma unroll
    for (int k = 0; k < NRED - 1; ++k) {
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = acc[(32 * k + i) / M][(32 * k + i) % M];
        warp_transpose_reduce<32>(v, lane);
        out[k] = v[0];
    }
    float v[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) {
        constexpr int dummy = 0;
        const int vi = LAST + i < V ? LAST + i : dummy;
        v[i] = LAST + i < V ? acc[vi / M][vi % M] : 0.0f;
    }
    warp_transpose_reduce<PL>(v, lane);
    out[NRED - 1] = v[0];
}

// Bulk prefetch of global memory into L2 (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

constexpr int RING_PREFETCH_JOBS = 6;  // jobs per warp prefetched into L2 beyond the ring's first S - 1

// A warp's copy stream (kept by lane 0): the next chunk's source, the chunk
// sizes of the current group (all but a row's last chunk, the last), the
// chunk, the item's end chunk and the item.
struct alignas(16) RingStream {
    const uint8_t* src;
    uint32_t cbr, cbl;
    int c, c1, it, pad;
};
static_assert(sizeof(RingStream) == 32, "RingStream is two 16-byte words");

// The row groups a ring kernel covers: those of one packed weight, or of two
// with the same K (the second's groups numbered after the first's), each
// with its own output.
// (Kernels of one weight do not use it: they read the kernel parameters.)
struct alignas(16) RowSpace {
    const uint8_t* w0;
    const uint8_t* w1;
    float* y0;
    float* y1;
    int64_t G0;  // groups of the first weight
    int N0, N1;
    __device__ __forceinline__ bool second(int64_t g) const { return g >= G0; }
    __device__ __forceinline__ int rows(int64_t g) const
    {
        const int64_t r = !second(g) ? (int64_t)N0 - g * GROUP : (int64_t)N1 - (g - G0) * GROUP;
        return r < GROUP ? (int)r : GROUP;
    }
    __device__ __forceinline__ const uint8_t* group_src(int64_t g, int64_t GB) const
    {
        return !second(g) ? w0 + g * GB : w1 + (g - G0) * GB;
    }
    __device__ __forceinline__ float* y_of(int64_t g) const { return !second(g) ? y0 : y1; }
    __device__ __forceinline__ int64_t local(int64_t g) const { return !second(g) ? g : g - G0; }
};

// sp: the pair's row space, or null for one weight at `base`.
template <bool PAIR>
__device__ __forceinline__ void ring_stream_at(RingStream& k, const RowSpace* sp, const uint8_t* base, const Layout& L,
                                               int64_t g0, int n_items, int P, uint32_t CB, uint32_t CBL, int64_t GB,
                                               int it)
{
    k.it = it;
    if (it >= n_items) return;
    const int q = P == 1 ? it : it / P;
    const int p = it - q * P;
    const int64_t g = g0 + q;
    const int rows = PAIR ? sp->rows(g) : L.rows_in(g);
    k.c = P == 1 ? 0 : p * L.nch / P;
    k.c1 = P == 1 ? L.nch : (p + 1) * L.nch / P;
    k.cbr = rows == GROUP ? CB : (uint32_t)L.chunk_bytes(rows, 0);
    k.cbl = rows == GROUP ? CBL : (uint32_t)L.chunk_bytes(rows, L.nch - 1);
    k.src = (PAIR ? sp->group_src(g, GB) : base + g * GB) + (int64_t)k.c * k.cbr;
}

// Loads of one 4-row group's chunk from a ring stage.  whole: 4 rows and 32
// blocks (compile-time offsets); otherwise `rows` rows and nb blocks (lanes
// >= nb are idle): rows past the group's end repeat its last row (Q4_0) or
// read stale bytes of the stage (Q6_K); their sums are discarded.
template <int FMT>
struct HalfLoads;

template <>
struct HalfLoads<FMT_Q4_0> {
    uint4 w16[R_ROWS];
    float dw[R_ROWS];
    __device__ __forceinline__ void whole(const uint8_t* st, int lane)
    {
#pragma unroll
        for (int q = 0; q < R_ROWS; ++q) w16[q] = *reinterpret_cast<const uint4*>(st + q * (CHUNK * 16) + lane * 16);
        const uint2 dd = *reinterpret_cast<const uint2*>(st + R_ROWS * CHUNK * 16 + lane * 8);
        dw[0] = __half2float(__ushort_as_half((unsigned short)(dd.x & 0xFFFFu)));
        dw[1] = __half2float(__ushort_as_half((unsigned short)(dd.x >> 16)));
        dw[2] = __half2float(__ushort_as_half((unsigned short)(dd.y & 0xFFFFu)));
        dw[3] = __half2float(__ushort_as_half((unsigned short)(dd.y >> 16)));
    }
    __device__ __forceinline__ void part(const uint8_t* st, int lane, int rows, int nb)
    {
#pragma unroll
        for (int q = 0; q < R_ROWS; ++q) {
            const int rq = min(q, rows - 1);
            w16[q] = *reinterpret_cast<const uint4*>(st + (rq * nb + lane) * 16);
            dw[q] = __half2float(
                __ushort_as_half(*reinterpret_cast<const uint16_t*>(st + nb * rows * 16 + (lane * rows + rq) * 2)));
        }
    }
};

template <>
struct HalfLoads<FMT_Q6_K> {
    uint4 cp[R_ROWS];
    uint2 cq[R_ROWS];
    uint32_t sc[R_ROWS];
    float dw[R_ROWS];
    __device__ __forceinline__ void whole(const uint8_t* st, int lane)
    {
        constexpr int TB = CHUNK * 26;
#pragma unroll
        for (int q = 0; q < R_ROWS; ++q) {
            cp[q] = *reinterpret_cast<const uint4*>(st + q * TB + lane * 16);
            cq[q] = *reinterpret_cast<const uint2*>(st + q * TB + CHUNK * 16 + lane * 8);
            sc[q] = *reinterpret_cast<const uint16_t*>(st + q * TB + CHUNK * 24 + lane * 2);
            dw[q] = __half2float(__ushort_as_half(
                *reinterpret_cast<const uint16_t*>(st + R_ROWS * TB + (q * (CHUNK / 8) + (lane >> 3)) * 2)));
        }
    }
    __device__ __forceinline__ void part(const uint8_t* st, int lane, int rows, int nb)
    {
        const int tb = nb * 26;
        const uint16_t* dq = reinterpret_cast<const uint16_t*>(st + rows * tb);
#pragma unroll
        for (int q = 0; q < R_ROWS; ++q) {
            cp[q] = *reinterpret_cast<const uint4*>(st + q * tb + lane * 16);
            cq[q] = *reinterpret_cast<const uint2*>(st + q * tb + nb * 16 + lane * 8);
            sc[q] = *reinterpret_cast<const uint16_t*>(st + q * tb + nb * 24 + lane * 2);
            dw[q] = __half2float(__ushort_as_half(dq[min(q, rows - 1) * (nb >> 3) + (lane >> 3)]));
        }
    }
};

// One lane's block of a 4-row group against the tile.
template <int M>
__device__ __forceinline__ void ring_dot4(const HalfLoads<FMT_Q4_0>& H, const uint8_t* ab, const uint8_t* am,
                                          float (&acc)[R_ROWS][M])
{
    uint32_t w[R_ROWS][8];
#pragma unroll
    for (int q = 0; q < R_ROWS; ++q) q4_0_unpack(H.w16[q], w[q]);
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 lo = *reinterpret_cast<const uint4*>(ab + 32 * m);
        const uint4 hi = *reinterpret_cast<const uint4*>(ab + 32 * m + 16);
        const uint2 mt = *reinterpret_cast<const uint2*>(am + 8 * m);
        const float da = __uint_as_float(mt.x);
#pragma unroll
        for (int q = 0; q < R_ROWS; ++q) {
            const int sI = q4_0_dot(w[q], lo, hi, (int)mt.y);
            acc[q][m] = fmaf(H.dw[q] * da, __int_as_float(sI) - MAGIC_I2F, acc[q][m]);
        }
    }
}

template <int M>
__device__ __forceinline__ void ring_dot4(const HalfLoads<FMT_Q6_K>& H, const uint8_t* ab, const uint8_t* am,
                                          float (&acc)[R_ROWS][M])
{
    uint32_t w[R_ROWS][8];
    int sc0x4[R_ROWS], sc1[R_ROWS];
    float dq[R_ROWS];  // the superblock scale over four (q6_k_dot_init returns 4 J)
#pragma unroll
    for (int q = 0; q < R_ROWS; ++q) {
        q6_k_unpack(H.cp[q], H.cq[q], w[q]);
        sc0x4[q] = 4 * (int)(int8_t)(H.sc[q] & 0xFFu);
        sc1[q] = (int)(int8_t)((H.sc[q] >> 8) & 0xFFu);
        dq[q] = H.dw[q] * 0.25f;
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 lo = *reinterpret_cast<const uint4*>(ab + 32 * m);
        const uint4 hi = *reinterpret_cast<const uint4*>(ab + 32 * m + 16);
        const uint4 mt = *reinterpret_cast<const uint4*>(am + 16 * m);
        const float da = __uint_as_float(mt.x);
#pragma unroll
        for (int q = 0; q < R_ROWS; ++q) {
            const int J4 = q6_k_dot_init(w[q], lo, hi, (int)mt.y, (int)mt.z, sc0x4[q], sc1[q]);
            acc[q][m] = fmaf(dq[q] * da, (float)J4, acc[q][m]);
        }
    }
}

template <int FMT, int M, bool TOP1, bool PAIR, bool RES = false, bool TOPK = false>
__global__ void __launch_bounds__(MmvqThreads<FMT, M, TOP1, TOPK>::value, 1)
    mmvq_ring_kernel(const MmvqArgs a, unsigned int* timeouts)
{
    static_assert(!TOPK || (TOP1 && !PAIR && !RES), "top-k is a top-1 kernel of one weight");
    constexpr int R = R_ROWS;
    constexpr int V = R * M;              // sums per row group
    constexpr int NRED = (V + 31) / 32;   // reduced sums per lane
    using Act = RingAct<FMT, M>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, W = blockDim.x >> 5;
    const int warp = __shfl_sync(0xffffffffu, (int)(threadIdx.x >> 5), 0);  // warp-uniform
    const int S = a.stages, P = a.parts;
    const Layout L = make_layout(FMT, a.N, a.K);
    const int NB = L.NB, nch = L.nch;
    const uint32_t CB = (uint32_t)L.chunk_bytes(R, 0), CBL = (uint32_t)L.chunk_bytes(R, nch - 1);
    pdl_launch_dependents();
    const int64_t GB = L.group_bytes(R);
    // A pair's row space lives in shared memory (read where needed), so that
    // it holds no registers in the main loop; one weight uses the kernel
    // parameters themselves.
    RowSpace* sp = PAIR ? reinterpret_cast<RowSpace*>(smem) : nullptr;
    if (PAIR && threadIdx.x == 0) {
        sp->w0 = static_cast<const uint8_t*>(a.w_pack);
        sp->w1 = static_cast<const uint8_t*>(a.w_pack2);
        sp->y0 = a.y;
        sp->y1 = a.y2;
        sp->G0 = L.n_groups;
        sp->N0 = a.N;
        sp->N1 = a.N2;
    }
    const uint8_t* wbase = static_cast<const uint8_t*>(a.w_pack);
    const int64_t n_groups = L.n_groups + (PAIR ? ((int64_t)a.N2 + GROUP - 1) / GROUP : 0);
    const int64_t g0 = (int64_t)blockIdx.x * n_groups / gridDim.x;
    const int64_t g1 = (int64_t)(blockIdx.x + 1) * n_groups / gridDim.x;
    const int ng = (int)(g1 - g0);
    const int n_items = ng * P;

    constexpr size_t SP_BYTES = PAIR ? sizeof(RowSpace) : 0;
    RingStream* streams = reinterpret_cast<RingStream*>(smem + SP_BYTES);  // [W], 16-byte aligned
    uint8_t* rings = smem + SP_BYTES + (size_t)W * sizeof(RingStream);
    Act t;
    t.q = rings + (size_t)W * S * CB;
    t.meta = t.q + (size_t)NB * Act::QSTRIDE;
    uint64_t* bars = reinterpret_cast<uint64_t*>(t.meta + (size_t)NB * Act::MROWS * Act::META);
    float* part = reinterpret_cast<float*>(bars + W * S);
    unsigned long long* s_best = reinterpret_cast<unsigned long long*>(part + (P > 1 ? (size_t)ng * P * V : 0));
    int* s_last = reinterpret_cast<int*>(s_best + MAX_M);
    // top-1: running key of each reduced sum a lane holds, [NRED][W * 32]
    unsigned long long* s_lane_best = reinterpret_cast<unsigned long long*>(s_best + MAX_M + 2);
    // top-k: the warps' lists, [W][M][TOPK_MAX]
    unsigned long long* s_topk = s_lane_best + (size_t)NRED * W * 32;
    const int KT = TOPK ? (int)a.topk : 0;  // k of the top-k
    static_assert(Act::META % 8 == 0 && (V * sizeof(float)) % 8 == 0, "ring shared-memory alignment");

    uint64_t* wbar = bars + warp * S;
    uint8_t* wring = rings + (size_t)warp * S * CB;
    const uint64_t pol = l2_evict_first_policy();
#ifdef QGEMV_BOUNDS_CHECK
    {
        // (debug build: the layout above must end within the launch's shared memory)
        const uint8_t* end = TOP1 ? reinterpret_cast<const uint8_t*>(s_topk + (TOPK ? (size_t)W * M * TOPK_MAX : 0))
                                  : reinterpret_cast<const uint8_t*>(part + (P > 1 ? (size_t)ng * P * V : 0));
        if (!QG_OK(end - smem <= (ptrdiff_t)dynamic_smem_bytes() && warp < W, timeouts, 610)) return;
    }
#endif

    if (TOP1) {
        if (threadIdx.x < MAX_M) s_best[threadIdx.x] = 0ull;
#pragma unroll
        for (int j = 0; j < NRED; ++j) s_lane_best[j * blockDim.x + threadIdx.x] = 0ull;
    }
    if (TOPK) {
        for (int i = lane; i < M * TOPK_MAX; i += 32) s_topk[(size_t)warp * M * TOPK_MAX + i] = 0ull;
    }
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&wbar[s], 1);
        fence_barrier_init();
    }
    if (PAIR) __syncthreads();  // the row space is visible to every warp
    else __syncwarp();

    // Lane 0's copy stream, kept in shared memory so that it holds no
    // registers in the main loop.
    RingStream& k = streams[warp];
    if (lane == 0) ring_stream_at<PAIR>(k, sp, wbase, L, g0, n_items, P, CB, CBL, GB, warp);
    // The next item is usually the whole group W groups on (P = 1) of the
    // same weight: its first chunk starts (W - 1) * GB past the end of the
    // current group.
    const int64_t skip = (int64_t)(W - 1) * GB;
    const int64_t last_whole = (a.N % GROUP) ? L.n_groups - 2 : L.n_groups - 1;  // one weight: its last full group
    // Lane 0 takes the next job off its stream (bytes = 0: none left).
    auto next_job = [&](const uint8_t*& src) -> uint32_t {
        RingStream ks = k;  // one copy in, one copy out
        if (ks.it >= n_items) return 0;
        const uint32_t bytes = ks.c == nch - 1 ? ks.cbl : ks.cbr;
        src = ks.src;
        ks.src += bytes;
        if (++ks.c == ks.c1) {
            const int nit = ks.it + W;
            // next group whole and of the same weight
            const bool next_whole = PAIR ? sp->rows(g0 + nit) == GROUP && sp->second(g0 + nit) == sp->second(g0 + ks.it)
                                         : g0 + nit <= last_whole;
            if (P == 1 && ks.cbr == CB && nit < n_items && next_whole) {
                ks.src += skip;
                ks.c = 0;
                ks.it = nit;
            } else {
                ring_stream_at<PAIR>(ks, sp, wbase, L, g0, n_items, P, CB, CBL, GB, nit);
            }
        }
        k = ks;
        return bytes;
    };
    // The whole warp: the copy's operands are made warp-uniform (broadcast
    // from lane 0, slot counted by every lane) and lane 0 issues it.
    int issued = 0, iss_slot = 0;
    const uint64_t pol_u = __shfl_sync(0xffffffffu, pol, 0);
    auto issue_next = [&]() {
        const uint8_t* src = wbase;
        uint32_t bytes = 0;
        if (lane == 0) bytes = next_job(src);
        bytes = __shfl_sync(0xffffffffu, bytes, 0);
        if (bytes == 0) return;
        src = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src), 0));
        uint64_t* bar = wbar + iss_slot;
        if (lane == 0) {
            fence_proxy_async();
            // (debug build: a copy outside the packs is skipped, its stage completing empty)
            const bool ok = QG_OK(pack_range_ok(a, FMT, src, bytes) && bytes <= CB, timeouts, 601);
            mbar_arrive_expect_tx(bar, ok ? bytes : 0u);
            if (ok) bulk_g2s(wring + (size_t)iss_slot * CB, src, bytes, bar, pol_u);
        }
        ++issued;
        if (++iss_slot == S) iss_slot = 0;
    };
    // Common case (one weight, P = 1, all groups whole, S <= nch): the copy
    // S - 1 jobs ahead of job (item it, chunk c) follows from it and c alone,
    // which every lane knows, so no stream state is read or written.
    const bool direct = !PAIR && P == 1 && (a.N % GROUP) == 0 && S <= nch;
    auto issue_direct = [&](int it, int c) {
        int ci = c + S - 1, iti = it;
        if (ci >= nch) {
            ci -= nch;
            iti += W;
        }
        if (iti >= n_items) return;
        const uint32_t bytes = ci == nch - 1 ? CBL : CB;
        const uint8_t* src = wbase + (g0 + iti) * GB + (int64_t)ci * CB;
        uint64_t* bar = wbar + iss_slot;
        if (lane == 0) {
            fence_proxy_async();
            const bool ok = QG_OK(pack_range_ok(a, FMT, src, bytes) && bytes <= CB, timeouts, 602);
            mbar_arrive_expect_tx(bar, ok ? bytes : 0u);
            if (ok) bulk_g2s(wring + (size_t)iss_slot * CB, src, bytes, bar, pol_u);
        }
        ++issued;
        if (++iss_slot == S) iss_slot = 0;
    };
    if (lane == 0) {
        // Start HBM on the first jobs (L2 prefetch) while the previous kernel
        // of the stream drains and the activation is staged.
        RingStream pf = k;
        for (int j = 0; j < S - 1 + RING_PREFETCH_JOBS && pf.it < n_items; ++j) {
            const uint32_t bytes = pf.c == nch - 1 ? pf.cbl : pf.cbr;
            if (QG_OK(pack_range_ok(a, FMT, pf.src, bytes), timeouts, 603)) bulk_prefetch_l2(pf.src, bytes);
            pf.src += bytes;
            if (++pf.c == pf.c1) ring_stream_at<PAIR>(pf, sp, wbase, L, g0, n_items, P, CB, CBL, GB, pf.it + W);
        }
    }
    pdl_wait();  // the previous kernel's writes (activation, weights, workspace) are visible from here
    for (int s = 0; s < S - 1; ++s) issue_next();

    if (!TOP1 || a.xq) ring_act_from_q8_1<FMT, M>(t, a.xq, NB);
    else ring_act_from_f32<FMT, M>(t, a.x, a.ldx, NB);
    __syncthreads();

    int consumed = 0, slot = 0;
    uint32_t phase = 0;
    bool alive = true;
    // item it = (group gl, part p); it -> it + W moves (gl, p) by (W / P, W % P)
    const int step_g = W / P, step_p = W - (W / P) * P;
    int gl = warp / P, p = warp - (warp / P) * P;
    for (int it = warp; it < n_items; it += W) {
        if (FMT == FMT_Q4_0 && lane == 0 && it + 2 * W < n_items) {
            // keep the short Q4_0 rings fed from L2: prefetch this warp's
            // item after next (its chunks are one contiguous region) while
            // this one is worked on
            const int ia = it + 2 * W;
            const int qa = P == 1 ? ia : ia / P, pa = ia - qa * P;
            const int64_t ga = g0 + qa;
            if (PAIR ? sp->rows(ga) == GROUP : ga <= last_whole) {
                const int ca = P == 1 ? 0 : pa * nch / P, cb = P == 1 ? nch : (pa + 1) * nch / P;
                const uint32_t span = (uint32_t)(cb - ca) * CB - (cb == nch ? CB - CBL : 0u);
                const uint8_t* ps = (PAIR ? sp->group_src(ga, GB) : wbase + ga * GB) + (int64_t)ca * CB;
                if (QG_OK(pack_range_ok(a, FMT, ps, span), timeouts, 604)) bulk_prefetch_l2(ps, span);
            }
        }
        const int64_t g = g0 + gl;
        const int rows = PAIR ? sp->rows(g) : L.rows_in(g);
        float acc[R][M];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < M; ++m) acc[r][m] = 0.0f;
        const int c0 = P == 1 ? 0 : p * nch / P, c1 = P == 1 ? nch : (p + 1) * nch / P;
        for (int c = c0; c < c1; ++c) {
            if (direct) issue_direct(it, c);
            else issue_next();
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&wbar[slot], phase))) {
                if (lane == 0) atomicAdd_system(timeouts, 1u);
                alive = false;
                break;
            }
            ++consumed;
            const uint8_t* st = wring + (size_t)slot * CB;
            const int ti = c * CHUNK + lane;
            const uint8_t* ab = t.q + ti * Act::QSTRIDE;
            const uint8_t* am = t.meta + ti * (Act::MROWS * Act::META);
            HalfLoads<FMT> H;
            if (rows == R && (c != nch - 1 || L.nb_tail == CHUNK)) {
                H.whole(st, lane);
                ring_dot4<M>(H, ab, am, acc);
            } else {
                const int nb = L.nb(c);
                if (lane < nb) {
                    H.part(st, lane, rows, nb);
                    ring_dot4<M>(H, ab, am, acc);
                }
            }
            __syncwarp();
            if (++slot == S) {
                slot = 0;
                phase ^= 1u;
            }
        }
        if (!alive) break;

        float v[NRED];
        ring_reduce<M, R>(acc, v, lane);
        if (TOPK) {
            // (P == 1 and one weight here)
            unsigned long long key[NRED];
            int row[NRED];
#pragma unroll
            for (int j = 0; j < NRED; ++j) {
                const int vi = ring_value_index<V>(j, lane);
                const int rr = vi / M, m = vi - rr * M;
                const bool own = ring_value_owner<V>(j, lane) && rr < rows;
                const int n = (int)(g * GROUP) + rr;
                key[j] = own ? top1_key(v[j], n) : 0ull;
                row[j] = own ? m : 0;
                if (own && a.cand_vals && n == a.cand[m]) a.cand_vals[m] = v[j];
            }
            topk_offer<NRED>(s_topk + (size_t)warp * M * TOPK_MAX, KT, key, row, lane);
        }
#pragma unroll
        for (int j = 0; j < NRED; ++j) {
            if (TOPK) break;
            const int vi = ring_value_index<V>(j, lane);
            if (!ring_value_owner<V>(j, lane)) continue;
            if (P > 1) {
                part[((size_t)gl * P + p) * V + vi] = v[j];
                continue;
            }
            const int rr = vi / M, m = vi - rr * M;
            if (rr < rows) {
                const int n = (int)((PAIR ? sp->local(g) : g) * GROUP) + rr;
                if (TOP1) {
                    // the lane's running key for value vi (chunk j of the reduction)
                    unsigned long long& b = s_lane_best[j * blockDim.x + threadIdx.x];
                    const unsigned long long key = top1_key(v[j], n);
                    if (key > b) b = key;
                    if (a.cand_vals && n == a.cand[m]) a.cand_vals[m] = v[j];
                } else {
                    float* y = PAIR ? sp->y_of(g) : a.y;
                    int64_t ns = n;
#ifdef QGEMV_BOUNDS_CHECK
                    if (a.plant_bad_store && blockIdx.x == 0 && warp == 0 && it == 0) ns += a.N;
#endif
                    if (QG_OK(store_ok(a, y, m, M, ns), timeouts, 620)) mmvq_store<RES>(a, y, m, ns, v[j]);
                }
            }
        }
        gl += step_g;
        p += step_p;
        if (p >= P) {
            p -= P;
            ++gl;
        }
    }
    // After a timeout, give the copies still in flight a bounded wait before
    // the shared memory is released.
    if (lane == 0) {
        for (int jj = consumed; jj < issued; ++jj) mbar_wait_bounded(&wbar[jj % S], (uint32_t)((jj / S) & 1));
    }
    __syncwarp();

    if (P > 1) {
        // Add the parts of every output in part order.
        __syncthreads();
        for (int o = threadIdx.x; o < ng * V; o += blockDim.x) {
            const int q = o / V, vi = o - q * V;
            const float* pp = part + (size_t)q * P * V + vi;
            float sum = pp[0];
            for (int j = 1; j < P; ++j) sum += pp[(size_t)j * V];
            const int rr = vi / M, m = vi - rr * M;
            const int64_t g = g0 + q;
            if (rr < (PAIR ? sp->rows(g) : L.rows_in(g))) {
                const int64_t n = (PAIR ? sp->local(g) : g) * GROUP + rr;
                if (TOP1) atomicMax(&s_best[m], top1_key(sum, (int)n));
                else if (QG_OK(store_ok(a, PAIR ? sp->y_of(g) : a.y, m, M, n), timeouts, 621))
                    mmvq_store<RES>(a, PAIR ? sp->y_of(g) : a.y, m, n, sum);
            }
        }
    }
    if (TOPK) {
        __syncthreads();  // every warp's lists are final
        // this CTA's k best keys per row, from the warps' lists
        for (int m = warp; m < M; m += W) {
            unsigned long long* dst = a.topk_lists + ((size_t)blockIdx.x * M + m) * KT;
            topk_select(
                W * KT, KT, lane,
                [&](int e) {
                    const int w = e / KT;
                    return s_topk[((size_t)w * M + m) * TOPK_MAX + (e - w * KT)];
                },
                [&](int r, unsigned long long key) { dst[r] = key; });
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            const unsigned prev = atomicAdd(&a.ws->done, 1u);
            *s_last = prev == gridDim.x - 1;
        }
        __syncthreads();
        if (*s_last) {
            __threadfence();
            // Merge the CTAs' lists ([CTA][row][k], each sorted larger
            // first): the row's warp copies its G lists (eight loads a lane
            // in flight) into the row's slice of the rings and the activation
            // tile, both free now, and merges them there (topk_merge_sorted).
            // Should they not fit, the k largest are picked from the lists in
            // global memory directly.
            const int G = gridDim.x;
            const unsigned long long* lists = a.topk_lists;
            unsigned long long* region = reinterpret_cast<unsigned long long*>(rings);
            const int total = G * KT;
            const bool fits = (size_t)M * total * 8 <= (size_t)(t.meta - rings) && G <= 32 * TOPK_HEADS;
            for (int m = warp; m < M; m += W) {
                auto emit = [&](int r, unsigned long long key) {
                    a.ids[m * KT + r] = key ? top1_key_to_id(key) : -1;
                    if (a.top_vals) a.top_vals[m * KT + r] = key ? top1_key_to_value(key) : __int_as_float(0x7fffffff);
                };
                if (!fits) {
                    topk_select(
                        total, KT, lane,
                        [&](int e) {
                            const int c = e / KT;
                            return __ldcg(lists + ((size_t)c * M + m) * KT + (e - c * KT));
                        },
                        emit);
                    continue;
                }
                unsigned long long* buf = region + (size_t)m * total;
#pragma unroll 8
                for (int e = lane; e < total; e += 32) {
                    const int c = e / KT;
                    buf[e] = __ldcg(lists + ((size_t)c * M + m) * KT + (e - c * KT));
                }
                __syncwarp();
                topk_merge_sorted(buf, G, KT, KT, lane, emit);
                __syncwarp();
            }
            if (threadIdx.x == 0) atomicExch(&a.ws->done, 0u);
        }
    }
    if (TOP1 && !TOPK) {
        if (P == 1) {
#pragma unroll
            for (int j = 0; j < NRED; ++j) {
                const unsigned long long b = s_lane_best[j * blockDim.x + threadIdx.x];
                if (b != 0ull) atomicMax(&s_best[ring_value_index<V>(j, lane) % M], b);
            }
        }
        __syncthreads();
        if (threadIdx.x < M) atomicMax(&a.ws->keys[threadIdx.x], s_best[threadIdx.x]);
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
                const unsigned long long key = atomicExch(&a.ws->keys[threadIdx.x], 0ull);
                a.ids[threadIdx.x] = top1_key_to_id(key);
                if (a.top_vals) a.top_vals[threadIdx.x] = top1_key_to_value(key);
            }
            if (threadIdx.x == 0) atomicExch(&a.ws->done, 0u);
        }
    }
}

// Shared memory of the ring kernel besides the rings, their mbarriers and
// the tile.
template <int M, bool TOP1, bool PAIR, bool TOPK = false>
inline size_t ring_extra_bytes(int max_groups_per_cta, int P, int warps)
{
    const size_t streams = (PAIR ? sizeof(RowSpace) : 0) + (size_t)warps * sizeof(RingStream);
    const size_t part = P > 1 ? (size_t)max_groups_per_cta * P * R_ROWS * M * sizeof(float) : 0;
    const size_t nred = (R_ROWS * M + 31) / 32;
    return streams + part + (TOP1 ? (size_t)(MAX_M + 2) * 8 + nred * warps * 32 * 8 : 0) +
           (TOPK ? (size_t)warps * M * TOPK_MAX * 8 : 0);
}

// ---------------------------------------------------------------------------
// Lock-step kernel: for activations too large for shared memory next to the
// rings.  K is staged in chunks of KC blocks (a multiple of 32); all warps
// move through the chunks together; weights are read with streaming loads.
//   shared memory: aq [M][2][KC] | am [M][KC] | TOP1 scratch
// ---------------------------------------------------------------------------

template <int FMT, int M, bool TOP1, bool RES = false>
__global__ void __launch_bounds__(MmvqThreads<FMT, M, TOP1>::value, 1)
    mmvq_lockstep_kernel(const MmvqArgs a, unsigned int* status)
{
    pdl_launch_dependents();
    pdl_wait();
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
    unsigned long long* s_best = s_keys + W * TOP1_GROUP_KEYS;
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
            if (!TOP1 || a.xq) stage_from_q8_1<FMT, M>(t, a.xq, NB, kb0, kb1);
            else stage_from_f32<FMT, M>(t, a.x, a.ldx, kb0, kb1);
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
                        if (!QG_OK(pack_range_ok(a, FMT, ad.q, 16) && pack_range_ok(a, FMT, ad.d, 2), status, 701)) {
                            w16[r] = make_uint4(0u, 0u, 0u, 0u);
                            dw[r] = 0.0f;
                            continue;
                        }
                        w16[r] = ld_stream_v4(reinterpret_cast<const uint4*>(ad.q));
                        dw[r] = __half2float(__ushort_as_half(ld_stream_u16(ad.d)));
                    }
                    accumulate_q4_0<M, R>(w16, dw, t, ti, acc);
                } else {
                    uint4 cp[R];
                    uint2 cq[R];
                    uint32_t sc[R];
                    float dw[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const BlockAddr ad = block_addr(a.w_pack, L, rows[r], b);
                        if (!QG_OK(pack_range_ok(a, FMT, ad.q, 16) && pack_range_ok(a, FMT, ad.qh, 8) &&
                                       pack_range_ok(a, FMT, ad.sc, 2) && pack_range_ok(a, FMT, ad.d, 2),
                                   status, 702)) {
                            cp[r] = make_uint4(0u, 0u, 0u, 0u);
                            cq[r] = make_uint2(0u, 0u);
                            sc[r] = 0u;
                            dw[r] = 0.0f;
                            continue;
                        }
                        cp[r] = ld_stream_v4(reinterpret_cast<const uint4*>(ad.q));
                        cq[r] = ld_stream_v2(reinterpret_cast<const uint2*>(ad.qh));
                        sc[r] = ld_stream_u16(ad.sc);
                        dw[r] = __half2float(__ushort_as_half(ld_stream_u16(ad.d)));
                    }
                    accumulate_q6_k<M, R>(cp, cq, sc, dw, t, ti, acc);
                }
            }
        }
        if (active)
            finish_rowgroup<M, R, TOP1, RES>(a, (int)(g * GROUP), acc, lane, s_keys + warp * TOP1_GROUP_KEYS, best,
                                             status);
    }
    if (TOP1) top1_finish<M>(a, s_best, s_last, best, lane, warp, W);
}

}  // namespace qgemv
