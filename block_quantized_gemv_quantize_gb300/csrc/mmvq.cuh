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
// Work decomposition (GB300, 152 SMs, one 512-thread CTA per SM):
//   * a warp owns a group of R consecutive weight rows and walks the whole K
//     dimension; lane l takes blocks b = l, l + 32, ... so that the 32 lanes
//     read 512 contiguous bytes of the packed nibble stream per row and load;
//   * each lane keeps R x M fp32 partial sums, reusing one activation block
//     (read from shared memory) for R rows and each weight block for M rows;
//   * a transpose-reduction sums the R x M partials over the 32 lanes with the
//     same butterfly tree for every output, so an output's value does not
//     depend on where its row sits (duplicated rows give identical floats);
//   * the activation tile (Q8_1 codes, fp16 scale, integer sums) is staged in
//     shared memory once per CTA; when it does not fit, K is processed in
//     chunks of a multiple of 32 blocks (same lane-to-block map, same order).
// Weights are streamed with L1-bypassing 16-byte loads and read exactly once.
#pragma once

#include "qgemv_common.cuh"

namespace qgemv {

constexpr int MMVQ_THREADS = 512;
constexpr int MMVQ_WARPS = MMVQ_THREADS / 32;

// Rows per warp for a given M: R * M partial sums per lane.
template <int M>
struct RowsPerWarp {
    static constexpr int value = M <= 8 ? 4 : 2;
};

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

// From fp32 activations, quantizing to Q8_1 on the fly (one warp per block),
// bit-identical to the standalone quantize_q8_1 kernel.
template <int FMT, int M>
__device__ __forceinline__ void stage_from_f32(const ActTile& t, const float* x, int64_t ldx, int kb0, int kb1)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int nbc = kb1 - kb0;
    int8_t* qbytes = reinterpret_cast<int8_t*>(t.aq);
    for (int i = warp; i < M * nbc; i += nw) {
        const int m = i / nbc, bl = i - m * nbc;
        const float xv = x[(int64_t)m * ldx + (int64_t)(kb0 + bl) * QK + lane];
        const Q81Lane r = q8_1_quantize_lane(xv);
        const int hsum = halfwarp_sum_i32(r.q);
        const int s1 = __shfl_sync(0xffffffffu, hsum, 16);
        qbytes[((m * 2 + (lane >> 4)) * t.KC + bl) * 16 + (lane & 15)] = (int8_t)r.q;
        if (lane == 0) {
            const float da = __half2float(__float2half_rn(r.d));
            uint2 meta;
            meta.x = __float_as_uint(da);
            meta.y = FMT == FMT_Q4_0 ? (uint32_t)(-8 * (hsum + s1))
                                     : (((uint32_t)hsum & 0xFFFFu) | ((uint32_t)s1 << 16));
            t.am[m * t.KC + bl] = meta;
        }
    }
}

// ---------------------------------------------------------------------------
// One row group over one K chunk.
// ---------------------------------------------------------------------------

template <int M, int R, int U>
__device__ __forceinline__ void rowgroup_chunk_q4_0(const PackQ40& pk, int NB, const int (&rows)[R], int kb0, int kb1,
                                                    const ActTile& t, int lane, float (&acc)[R][M])
{
    const uint4* nib[R];
    const __half* dsc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        nib[r] = pk.nib + (int64_t)rows[r] * NB;
        dsc[r] = pk.d + (int64_t)rows[r] * NB;
    }
    for (int b = kb0 + lane; b < kb1; b += 32 * U) {
        uint4 wv[U][R];
        uint16_t dh[U][R];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int bb = b + 32 * u;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (bb < kb1) {
                    wv[u][r] = ld_stream_v4(nib[r] + bb);
                    dh[u][r] = ld_stream_u16(dsc[r] + bb);
                } else {
                    wv[u][r] = make_uint4(0, 0, 0, 0);
                    dh[u][r] = 0;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int bb = b + 32 * u;
            if (bb < kb1) {
                const int ti = bb - kb0;
                uint32_t w[R][8];
                float dw[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    q4_0_unpack(wv[u][r], w[r]);
                    dw[r] = __half2float(__ushort_as_half(dh[u][r]));
                }
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
        }
    }
}

template <int M, int R, int U>
__device__ __forceinline__ void rowgroup_chunk_q6_k(const PackQ6K& pk, int NB, const int (&rows)[R], int kb0, int kb1,
                                                    const ActTile& t, int lane, float (&acc)[R][M])
{
    const int NSB = NB / 8;
    const uint4* ql[R];
    const uint2* qh[R];
    const uint16_t* sc[R];
    const __half* dd[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        ql[r] = pk.ql + (int64_t)rows[r] * NB;
        qh[r] = pk.qh + (int64_t)rows[r] * NB;
        sc[r] = pk.sc + (int64_t)rows[r] * NB;
        dd[r] = pk.d + (int64_t)rows[r] * NSB;
    }
    for (int b = kb0 + lane; b < kb1; b += 32 * U) {
        uint4 vl[U][R];
        uint2 vh[U][R];
        uint16_t vs[U][R], vd[U][R];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int bb = b + 32 * u;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (bb < kb1) {
                    vl[u][r] = ld_stream_v4(ql[r] + bb);
                    vh[u][r] = ld_stream_v2(qh[r] + bb);
                    vs[u][r] = ld_stream_u16(sc[r] + bb);
                    vd[u][r] = ld_stream_u16(dd[r] + (bb >> 3));
                } else {
                    vl[u][r] = make_uint4(0, 0, 0, 0);
                    vh[u][r] = make_uint2(0, 0);
                    vs[u][r] = 0;
                    vd[u][r] = 0;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int bb = b + 32 * u;
            if (bb < kb1) {
                const int ti = bb - kb0;
                uint32_t w[R][8];
                float dw[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    q6_k_unpack(vl[u][r], vh[u][r], w[r]);
                    dw[r] = __half2float(__ushort_as_half(vd[u][r]));
                }
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const uint4 lo = t.aq[(m * 2 + 0) * t.KC + ti];
                    const uint4 hi = t.aq[(m * 2 + 1) * t.KC + ti];
                    const uint2 mt = t.am[m * t.KC + ti];
                    const float da = __uint_as_float(mt.x);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const int J = q6_k_dot(w[r], lo, hi, mt.y, vs[u][r]);
                        acc[r][m] = fmaf(dw[r] * da, (float)J, acc[r][m]);
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// The kernel.
//   TOP1 = false: y[m * ldy + n] = result (activation from Q8_1 in xq).
//   TOP1 = true : activation quantized from fp32 x in the prologue; each row's
//                 greedy token id goes to ids[m]; no logits are written.
// ---------------------------------------------------------------------------

struct MmvqArgs {
    const void* w_pack;
    const uint8_t* xq;  // Q8_1 [M][NB] (TOP1 = false)
    const float* x;     // fp32 [M][ldx] (TOP1 = true)
    int64_t ldx;
    float* y;
    int64_t ldy;
    int K, N, KC;
    Top1Workspace* ws;
    int32_t* ids;
};

template <int FMT, int M, bool TOP1>
__global__ void __launch_bounds__(MMVQ_THREADS, 1) mmvq_kernel(const MmvqArgs a)
{
    constexpr int R = RowsPerWarp<M>::value;
    constexpr int V = R * M;
    constexpr int P = next_pow2(V);
    constexpr int C = P >= 32 ? P / 32 : 1;
    constexpr int U = FMT == FMT_Q4_0 ? 2 : 1;

    extern __shared__ uint4 smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int NB = a.K / QK;
    const int KC = a.KC;
    ActTile t;
    t.aq = smem;
    t.am = reinterpret_cast<uint2*>(smem + 2 * M * KC);
    t.KC = KC;
    unsigned long long* s_keys = reinterpret_cast<unsigned long long*>(t.am + M * KC);  // [warps][64]
    unsigned long long* s_best = s_keys + MMVQ_WARPS * 64;                               // [warps][MAX_M], flag

    const int n_rg = (a.N + R - 1) / R;
    const int n_items = (n_rg + MMVQ_WARPS - 1) / MMVQ_WARPS;
    const int nchunks = (NB + KC - 1) / KC;

    PackQ40 p4 = pack_q4_0(a.w_pack, a.N, NB);
    PackQ6K p6 = pack_q6_k(a.w_pack, a.N, NB);

    if (TOP1) {
        // Start this CTA's first weight rows on their way to L2 while the
        // activation is being quantized.
        const int rg = blockIdx.x * MMVQ_WARPS + warp;
        const int boff = (lane / R) * 32;  // one 512-byte segment per lane, inside the row
        if (rg < n_rg && boff < NB) {
            const int n = min(rg * R + (lane & (R - 1)), a.N - 1);
            if (FMT == FMT_Q6_K) prefetch_l2(p6.ql + (int64_t)n * NB + boff);
            else prefetch_l2(p4.nib + (int64_t)n * NB + boff);
        }
    }

    if (nchunks == 1) {
        if (TOP1) stage_from_f32<FMT, M>(t, a.x, a.ldx, 0, NB);
        else stage_from_q8_1<FMT, M>(t, a.xq, NB, 0, NB);
        __syncthreads();
    }

    unsigned long long best = 0ull;  // lane m < M: best key of row m seen by this warp

    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int rg = item * MMVQ_WARPS + warp;
        const bool active = rg < n_rg;
        const int n0 = rg * R;
        int rows[R];
#pragma unroll
        for (int r = 0; r < R; ++r) rows[r] = min(n0 + r, a.N - 1);

        float acc[R][M];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < M; ++m) acc[r][m] = 0.0f;

        for (int c = 0; c < nchunks; ++c) {
            const int kb0 = c * KC, kb1 = min(NB, kb0 + KC);
            if (nchunks > 1) {
                __syncthreads();
                if (TOP1) stage_from_f32<FMT, M>(t, a.x, a.ldx, kb0, kb1);
                else stage_from_q8_1<FMT, M>(t, a.xq, NB, kb0, kb1);
                __syncthreads();
            }
            if (active) {
                if (FMT == FMT_Q4_0) rowgroup_chunk_q4_0<M, R, U>(p4, NB, rows, kb0, kb1, t, lane, acc);
                else rowgroup_chunk_q6_k<M, R, U>(p6, NB, rows, kb0, kb1, t, lane, acc);
            }
        }
        if (!active) continue;

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
            unsigned long long* wk = s_keys + warp * 64;
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

    if (TOP1) {
        int& s_last = *reinterpret_cast<int*>(s_best + MMVQ_WARPS * MAX_M);
        if (lane < M) s_best[warp * MAX_M + lane] = best;
        __syncthreads();
        if (threadIdx.x < M) {
            unsigned long long k = 0ull;
            for (int w = 0; w < MMVQ_WARPS; ++w) {
                const unsigned long long kw = s_best[w * MAX_M + threadIdx.x];
                k = kw > k ? kw : k;
            }
            atomicMax(&a.ws->keys[threadIdx.x], k);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            const unsigned prev = atomicAdd(&a.ws->done, 1u);
            s_last = prev == gridDim.x - 1;
        }
        __syncthreads();
        if (s_last) {
            __threadfence();
            if (threadIdx.x < M) {
                const unsigned long long k = atomicExch(&a.ws->keys[threadIdx.x], 0ull);
                a.ids[threadIdx.x] = top1_key_to_id(k);
            }
            if (threadIdx.x == 0) atomicExch(&a.ws->done, 0u);
        }
    }
}

// Shared memory for one launch: activation tile + top-1 scratch.
template <int M, bool TOP1>
inline size_t mmvq_smem_bytes(int KC)
{
    size_t s = (size_t)M * KC * ACT_BYTES_PER_BLOCK;
    if (TOP1) s += (size_t)MMVQ_WARPS * 64 * 8 + (size_t)MMVQ_WARPS * MAX_M * 8 + 16;
    return s;
}

}  // namespace qgemv
