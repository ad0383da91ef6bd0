// Q4_0 x Q8_1 MMVQ on the tensor cores: exact per-block integer dots from
// f16 mma.sync (m16n8k16, fp32 accumulate), block scales applied in fp32.
//
// What is computed is exactly what the SIMT kernel computes ("Qwen3.6 27B
// Q4_0 DFlash/SYCL closure", What materially worked, item 2):
//     y[m][n] = sum_b fp16(d_w[n,b]) * fp16(d_a[m,b]) * I[m,n,b],
//     I[m,n,b] = sum_i (q_w[n,b,i] - 8) * q_a[m,b,i]   (an exact integer).
// Why tensor cores here: at M = 6 the dp4a formulation needs 48 dp4a per
// (row, block), and dp4a issues at half rate on this part, so the integer
// pipe alone takes as long as streaming the 18-byte block from HBM.  One
// m16n8k16 pair covers 16 rows x 32 values x 8 activation rows.
//
// Exactness.  The A operand (weights) is built from the 4-bit codes with one
// LOP3 per two values: f16 bits 0x6400 | q = 1024 + q (values 0..15 of the
// block's low nibbles) and 0x6400 | q << 4 = 1024 + 16 q (the high nibbles,
// whose B operand is staged as q_a / 16, exact in f16).  Every product is an
// integer (f16 x f16 is exact in fp32), and the accumulator is started at
//     C = -1032 * sum_{i<16} q_a - 72 * sum_{i>=16} q_a,
// so the MMA pair returns I exactly: all partial sums are integers below
// 2^23 in magnitude.  The scales are then applied per block in fp32:
//     y += (d_w * d_a) * I, summed per job of 8 blocks, then across jobs.
//
// Work decomposition (one CTA per SM, 16 warps):
//   * a tile is 16 weight rows (four 4-row groups of the packed layout); a
//     job is one tile x 16 blocks (4 KB of codes + 512 B of scales, three TMA
//     tensor copies), or x 8 blocks where shared memory is short; the code
//     boxes (8 blocks each) are 128-byte swizzled, so the 8 rows a warp reads
//     at once fall in distinct bank groups;
//   * a CTA owns a balanced, contiguous range of tiles and, in a cluster of C
//     CTAs, the C-th part of K (so only that part of the activation is staged);
//   * the CTA's jobs (tile-major) are cut into W equal contiguous ranges, one
//     per warp, each streaming through a private ring of S stages; a tile
//     that straddles two warps is summed from their pieces in warp order, and
//     the C parts of a tile in rank order (through distributed shared
//     memory), so the result does not depend on timing.
#pragma once

#include <cuda.h>

#include "mmvq.cuh"

namespace qgemv {

constexpr int TC_ROWS = 16;                     // weight rows per tile
constexpr int TC_LINE_JB = 8;                   // blocks per 128-byte line of a code box
constexpr int TC_BOX = TC_ROWS * TC_LINE_JB * 16;  // 2048 B: one code box (16 rows x 8 blocks)
// Blocks per job, chosen per launch: 16 (two code boxes, fewer jobs) where two
// ring stages of them fit next to the activation tile, else 8.
__host__ __device__ inline int tc_nib_bytes(int jb) { return TC_ROWS * jb * 16; }
__host__ __device__ inline int tc_ds_bytes(int jb) { return TC_ROWS * jb * 2; }
constexpr int TC_THREADS = 512;
// Weight formats of the tensor-core kernel: Q4_0 and Q6_K (the existing packs,
// read by tensor maps), Q8_0 and Q4_K (their own packs, one contiguous region
// per job).
enum TcFormat { TCF_Q4_0 = 0, TCF_Q6_K = 1, TCF_Q8_0 = 2, TCF_Q4_K = 3, TCF_Q5_K = 4 };
// A Q4_K job is one superblock (8 blocks) of a 16-row tile: codes [block
// p][lane 4g + t] 8 B (word t of row g's then of row g + 8's Q4_0-ordered
// 16 code bytes: byte k = value k | value k + 16 << 4), then [row][p] {scale,
// min} bytes (16 B per row), then [row] {fp16 d, fp16 dmin}.
constexpr int TC_Q4_K_JOB = 8 * 256 + 8 * TC_ROWS * 2 + TC_ROWS * 4;  // 2368 B
// Q5_K adds, after the codes, the fifth bits: [p][row] a 4-byte word whose
// byte k bit s is the fifth bit of value k + 4 s of block p.
constexpr int TC_Q5_K_JOB = TC_Q4_K_JOB + 8 * TC_ROWS * 4;  // 2880 B
// A Q6_K job is one superblock (8 blocks) of 16 rows: ring stage = ql box
// (16 x 128 B, 128-byte swizzle) + qh box (16 x 64 B, 64-byte swizzle), then
// in the scale ring the sc box (16 x 16 B) + the chunk's superblock scales
// (4 groups x 32 B).
constexpr int TC_Q6_K_NIB = TC_ROWS * 128 + TC_ROWS * 64;  // 3072 B
constexpr int TC_Q6_K_DS = TC_ROWS * 16 + 4 * 32;          // 384 B
constexpr int TC_Q8_0_CODES = TC_ROWS * 8 * 32;            // 4096 B: 16 rows x 8 blocks of int8 codes
constexpr int TC_Q8_0_JOB = TC_Q8_0_CODES + TC_ROWS * 8 * 2;  // + 256 B of scales = 4352 B
constexpr int TC_Q8_0_JOB_BLOCKS = 8;                          // blocks of a pack region
// ring-stage bytes of a Q8_0 job of jb blocks (8: a whole region; 4: half of
// its codes and half of its scales)
__host__ __device__ inline int tc_q8_0_job_bytes(int jb) { return jb * (512 + 32); }
constexpr int TC_MIN_M = 5;  // activation rows from which the tensor-core path is taken (Q4_0)
// below TC_MIN_M rows, the weight elements (N K, both weights of a pair) from
// which the small-M kernel is taken all the same (2^28: a 151 MB Q4_0 pack)
constexpr int64_t TC_SMALL_M_MIN_ELEMS = (int64_t)1 << 28;
constexpr int TC_Q6_K_MIN_M = 7;  // the same for Q6_K
constexpr int TC_MAX_STAGES = 6;

struct TcArgs {
    const uint8_t* xq;  // Q8_1 [M][NB]
    float* y;           // first weight's output
    float* y2;          // second weight's output (pairs)
    int64_t ldy;
    const float* res;   // optional residual, y = W x + res (one weight): [M][ldr], may be y
    int64_t ldr;
    const uint8_t* w0;  // Q8_0: the packed weights (the copies read them directly)
    const uint8_t* w1;
    int K, N, N2;       // Q4_0, Q6_K: N, N2 multiples of 16 and K of 1024; Q8_0: K a multiple of 256
    int stages;         // ring stages per warp
    int jb;             // blocks per job (8 or 16)
    int nkb_max;        // activation blocks staged per CTA (the largest K part)
    int out_tiles;      // clusters: tiles per cluster the result buffer holds
    int drop_copy;      // test only (small-M Q4_0 kernel): CTA 0's warp 0 issues no copy for its first job
};

// Shared-memory layout, identical on the host (sizing) and the device.
struct TcSmem {
    uint32_t nib, ds, act, meta, out, tab, bar, bytes;
};

constexpr int TC_TAB_INTS = 4 + 3 * (TC_THREADS / 32);  // the split-tile table

// meta bytes per (block, 8-row tile): {d_a, d_a', C, C'} per lane (64), the
// Q6_K pair of starts (128), or the Q4_K / Q5_K columns of d_a, C, d_a A (96)
__host__ __device__ constexpr int tc_meta_bytes(int fmt)
{
    return fmt == TCF_Q6_K ? 128 : (fmt == TCF_Q4_K || fmt == TCF_Q5_K) ? 96 : 64;
}

// nibs / dsb: bytes of a ring stage's codes / scales (Q8_0: the whole job / 0);
// metab: meta bytes per (block, 8-row tile): 64, or 128 for Q6_K (two
// accumulator starts)
__host__ __device__ inline TcSmem tc_smem(int M, int W, int S, int nkb, int out_tiles, int nibs, int dsb,
                                          int metab = 64)
{
    const uint32_t NT = (uint32_t)(M + 7) / 8;
    TcSmem s;
    uint32_t o = 0;
    s.nib = o;  o += (uint32_t)W * S * nibs;  // Q4_0: 1024-byte aligned stages (128-byte swizzle atoms)
    s.ds = o;   o += (uint32_t)W * S * dsb;
    s.act = o;  o += (uint32_t)nkb * M * 64;        // B fragments, [block][row][4 lanes] x 16 B
    s.meta = o; o += (uint32_t)nkb * NT * metab;    // [block][8-row tile][4 lanes] x {d_a, d_a, C, C (, C1, C1, -, -)}
    s.out = o;  o += (uint32_t)out_tiles * 32 * NT * 16;
    s.tab = o;  o += TC_TAB_INTS * 4;
    s.bar = o;  o += ((uint32_t)W * S + 1) * 8;     // ring barriers, then the activation's
    s.bytes = o + 1024;                              // room to align the base to 1024 B
    return s;
}

// ---------------------------------------------------------------------------
// PTX: TMA tensor copies, clusters, distributed shared memory, mma.sync.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar,
                                            uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// Bulk copy global -> shared without a cache hint (the activation, which
// every CTA reads).
__device__ __forceinline__ void bulk_g2s_plain(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster; shared-memory writes before it
// are visible to the cluster's reads after it.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Load a float from CTA `rank`'s shared memory at the address `p` has in ours.
__device__ __forceinline__ float ld_dsmem_f32(const float* p, uint32_t rank)
{
    uint32_t ra;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
    return v;
}

// D = A B + C, m16n8k16, f16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                              float c0, float c1, float c2, float c3)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

// f16x2 of (1024 + nibble) from bits 0..3 of each 16-bit half of v (mask
// 0x000F000F), or of (1024 + 16 nibble) from bits 4..7 (mask 0x00F000F0).
template <uint32_t MASK>
__device__ __forceinline__ uint32_t nib_f16x2(uint32_t v)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "n"(MASK), "n"(0x64006400));  // (v & MASK) | 0x6400..
    return r;
}

// ---------------------------------------------------------------------------
// Activation staging: the CTA's K part of the Q8_1 activation as B fragments.
// Lane (g, t) of an m16n8k16 holds B[k][n = g] for k = 2t, 2t+1 (register 0)
// and k = 2t+8, 2t+9 (register 1).  The K order inside a block is chosen to
// match the code unpacking (one 4-byte word per lane and row):
//   first MMA:  k = 2t, 2t+1   <- values 4t, 4t+2;   k = 2t+8, 2t+9 <- 4t+1, 4t+3
//   second MMA: the same with values 16 + ..., staged as q_a / 16.
// Block b, row n: 4 x 16 B at act + ((b * M + n) * 4 + t) * 16.
// Meta of block b, 8-row tile nt, lane t (rows 8 nt + 2t, + 1):
//   {d_a, d_a', C, C'} at meta + ((b * NT + nt) * 4 + t) * 16, zero for rows >= M.
// ---------------------------------------------------------------------------

// (block, row slot) items of the activation conversion per thread (four
// threads each): the plan keeps nkb * NT * 8 within tc_stage_items(M) *
// TC_THREADS (K = 5120 fits in one CTA up to M = 12).
__host__ __device__ constexpr int tc_stage_items(int M) { return M > 8 ? 6 : 4; }

// Bytes 0, 2 (sel 0x4240) or 1, 3 (sel 0x4341) of the int8 word w as f16x2,
// scaled by 1 or 1/16, exactly: (w ^ 0x80) is q + 128, and the f16 with bits
// 0x6400 | (q + 128) is 1024 + 128 + q.
template <uint32_t SEL, bool SIXTEENTH>
__device__ __forceinline__ uint32_t q8_f16x2(uint32_t w)
{
    const uint32_t b = __byte_perm(w ^ 0x80808080u, 0x64646464u, SEL);
    const __half2 h = *reinterpret_cast<const __half2*>(&b);
    const __half2 r = SIXTEENTH ? __hfma2(h, __float2half2_rn(0.0625f), __float2half2_rn(-72.0f))
                                : __hsub2(h, __float2half2_rn(1152.0f));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// raw: the K part's Q8_1 blocks in shared memory, row n's at raw + n * rstride
// (rstride = nkb * 36 + 16: the pad puts the rows in distinct bank groups),
// lying in the tail of the act region.  Thread item (block b, row n, lane t),
// t fastest, then n: phase 1 reads the lane's two code words (and the meta is
// written), phase 2, after every raw byte has been read, writes the lane's
// 16-byte B fragment; both are free of bank conflicts.
// FMT = TCF_Q6_K: the meta is 32 B per lane, {d_a, d_a', C0, C0', C1, C1', 0,
// 0} with the two MMAs' own starts, C0 = -1056 sum_{i<16} q_a (codes 1024 + q
// against q_a: (q - 32) q_a = (1024 + q) q_a - 1056 q_a) and C1 = -96
// sum_{i>=16} q_a (codes 1024 + 16 q against q_a / 16: 64 q_a + q q_a - 96 q_a).
// FMT = TCF_Q4_K / TCF_Q5_K: 96 B per (block, 8-row tile), [d_a x 8][C x
// 8][d_a A x 8] by column, with C = -1024 sum_{i<16} q_a - 64 sum_{i>=16} q_a
// (no code offset) and A = sum q_a (the min term; d_a A is exact in fp32).
template <int M, int FMT = TCF_Q4_0>
__device__ __forceinline__ void tc_stage_act(uint8_t* act, float* meta, const uint8_t* raw, int nkb, int rstride)
{
    constexpr int NT = (M + 7) / 8;
    constexpr int IT = 4 * tc_stage_items(M);
    const int total = nkb * NT * 32;
    uint32_t w0[IT], w1[IT];
#pragma unroll
    for (int u = 0; u < IT; ++u) {
        const int i = threadIdx.x + u * TC_THREADS;
        w0[u] = w1[u] = 0;
        if (i >= total) break;  // warp-uniform: total is a multiple of 32
        const int tt = i & 3, n = ((i >> 5) % NT) * 8 + ((i >> 2) & 7), b = (i >> 5) / NT;
        float da = 0.0f;
        if (n < M) {
            const uint8_t* blk = raw + (size_t)n * rstride + (size_t)b * Q8_1_BYTES;
            w0[u] = *reinterpret_cast<const uint32_t*>(blk + 4 + 4 * tt);
            w1[u] = *reinterpret_cast<const uint32_t*>(blk + 20 + 4 * tt);
            if (tt == 0) da = __half2float(*reinterpret_cast<const __half*>(blk));
        }
        int s_lo = __dp4a((int)w0[u], 0x01010101, 0), s_hi = __dp4a((int)w1[u], 0x01010101, 0);
        s_lo += __shfl_xor_sync(0xffffffffu, s_lo, 1);
        s_hi += __shfl_xor_sync(0xffffffffu, s_hi, 1);
        s_lo += __shfl_xor_sync(0xffffffffu, s_lo, 2);
        s_hi += __shfl_xor_sync(0xffffffffu, s_hi, 2);
        if (tt == 0) {
            const int nt = n >> 3, c = n & 7;
            if constexpr (FMT == TCF_Q6_K) {
                float* mp = meta + (((size_t)b * NT + nt) * 4 + (c >> 1)) * 8;
                mp[c & 1] = da;
                mp[2 + (c & 1)] = (float)(-1056 * s_lo);
                mp[4 + (c & 1)] = (float)(-96 * s_hi);
                mp[6 + (c & 1)] = 0.0f;
            } else if constexpr (FMT == TCF_Q4_K || FMT == TCF_Q5_K) {
                float* mp = meta + ((size_t)b * NT + nt) * 24;  // [d_a x 8][C x 8][d_a A x 8]
                mp[c] = da;
                mp[8 + c] = (float)(-1024 * s_lo - 64 * s_hi);
                mp[16 + c] = da * (float)(s_lo + s_hi);
            } else {
                float* mp = meta + (((size_t)b * NT + nt) * 4 + (c >> 1)) * 4;
                mp[c & 1] = da;
                mp[2 + (c & 1)] = (float)(-1032 * s_lo - 72 * s_hi);
            }
        }
    }
    __syncthreads();  // the raw bytes are all read
#pragma unroll
    for (int u = 0; u < IT; ++u) {
        const int i = threadIdx.x + u * TC_THREADS;
        if (i >= total) break;
        const int tt = i & 3, n = ((i >> 5) % NT) * 8 + ((i >> 2) & 7), b = (i >> 5) / NT;
        if (n >= M) continue;
        uint4 v;  // lane t's registers: values 4t, 4t+2 | 4t+1, 4t+3 | and the same + 16 (scaled)
        v.x = q8_f16x2<0x4240u, false>(w0[u]);
        v.y = q8_f16x2<0x4341u, false>(w0[u]);
        v.z = q8_f16x2<0x4240u, true>(w1[u]);
        v.w = q8_f16x2<0x4341u, true>(w1[u]);
        *reinterpret_cast<uint4*>(act + (((size_t)b * M + n) * 4 + tt) * 16) = v;
    }
}

// One job: 16 blocks of the tile in ring stage (sn codes, sd scales) against
// staged blocks kb .. kb + 7.  acc[nt][i]: rows g, g, g+8, g+8 and columns
// 8 nt + 2t, +1, +0, +1 (the mma accumulator layout).
template <int M>
__device__ __forceinline__ void tc_job(const uint8_t* sn, const uint8_t* sd, const uint8_t* act, const float* meta,
                                       int kb, int jb, int g, int t, float (&acc)[(M + 7) / 8][4])
{
    constexpr int NT = (M + 7) / 8;
    float jacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) jacc[nt][i] = 0.0f;
    // codes: box h (blocks 8h .. 8h + 7) at sn + 2048 h, row g in line g,
    // row g + 8 1024 B on; scales: [group][16 blocks][4 rows]
    const uint8_t* rg = sn + g * 128 + 4 * t;
    const uint8_t* dg = sd + (g >> 2) * (jb * 8) + (g & 3) * 2;  // row g + 8's are 2 groups on
#pragma unroll 1
    for (int p0 = 0; p0 < jb; p0 += TC_LINE_JB)  // one code box at a time
#pragma unroll
    for (int pp = 0; pp < TC_LINE_JB; ++pp) {
        const int p = p0 + pp;
        const int sw = (pp ^ g) << 4;  // 16-byte piece pp of line L sits at piece pp ^ (L & 7)
        const uint8_t* rp = rg + (p0 / TC_LINE_JB) * TC_BOX;
        const uint32_t wa = *reinterpret_cast<const uint32_t*>(rp + sw);
        const uint32_t wb = *reinterpret_cast<const uint32_t*>(rp + 1024 + sw);
        const float dwa = __half2float(*reinterpret_cast<const __half*>(dg + p * 8));
        const float dwb = __half2float(*reinterpret_cast<const __half*>(dg + 2 * jb * 8 + p * 8));
        const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
        const uint32_t A0[4] = {nib_f16x2<0x000F000Fu>(wa), nib_f16x2<0x000F000Fu>(wb), nib_f16x2<0x000F000Fu>(wa8),
                                nib_f16x2<0x000F000Fu>(wb8)};
        const uint32_t A1[4] = {nib_f16x2<0x00F000F0u>(wa), nib_f16x2<0x00F000F0u>(wb), nib_f16x2<0x00F000F0u>(wa8),
                                nib_f16x2<0x00F000F0u>(wb8)};
        const int b = kb + p;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int n = nt * 8 + g < M ? nt * 8 + g : M - 1;  // rows past M: any staged row (unused)
            const uint4 B = *reinterpret_cast<const uint4*>(act + (((size_t)b * M + n) * 4 + t) * 16);
            const float4 md = *reinterpret_cast<const float4*>(meta + (((size_t)b * NT + nt) * 4 + t) * 4);
            float d[4];
            mma_f16_16816(d, A0, B.x, B.y, md.z, md.w, md.z, md.w);
            mma_f16_16816(d, A1, B.z, B.w, d[0], d[1], d[2], d[3]);
            // jacc += (d_w d_a) D, the exact fp16 x fp16 product first
            float sa0, sa1, sb0, sb1;
            mul_f32x2(sa0, sa1, dwa, dwa, md.x, md.y);
            mul_f32x2(sb0, sb1, dwb, dwb, md.x, md.y);
            fma_f32x2(jacc[nt][0], jacc[nt][1], sa0, sa1, d[0], d[1]);
            fma_f32x2(jacc[nt][2], jacc[nt][3], sb0, sb1, d[2], d[3]);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] += jacc[nt][i];
}

// ---------------------------------------------------------------------------
// Q6_K over the existing pack (a row's chunk tile: P[32 blocks][16 B], then
// Q[32][8 B], then sc[32][2 B]; the chunk's superblock scales d[4 rows][4]
// after the four tiles).  Block value v < 16 is bits 0-5 of P byte v; value
// 16 + u has its high two bits at bits 6-7 of P byte u and its low four bits
// in Q byte u % 8 (bits 0-3 for u < 8, bits 4-7 for u >= 8).  Lane t takes
// values 4t .. 4t+3 and 16 + 4t .. 16 + 4t + 3 (the K order the activation
// is staged in): one P word and one Q word per row and block, the Q word
// shifted left by 4 for t < 2 so that the low four bits of value 16 + 4t + j
// sit at bits 4-7 of byte j.
// ---------------------------------------------------------------------------

// Two codes of the first half-block as an f16x2 A register: 1024 + q per
// half (the code's six bits under 0x6400), exactly.
__device__ __forceinline__ uint32_t q6_lo_f16x2(uint32_t p)
{
    return (p & 0x003F003Fu) | 0x64006400u;
}

// Two codes of the second half-block: 1024 + 16 q per half, the high two bits
// (h, already at bits 8-9) and the low four (l, at bits 4-7) under 0x6400.
__device__ __forceinline__ uint32_t q6_hi_f16x2(uint32_t h, uint32_t l)
{
    return (h & 0x03000300u) | (l & 0x00F000F0u) | 0x64006400u;
}

// Four-bit codes with a fifth bit as two f16x2 A registers per MMA (Q5_K):
// (lo & LO) | (hi & HM) | 0x6400 per half = 1024 + q (LO = 0x000F000F, HM =
// 0x00100010) or 1024 + 16 q (LO = 0x00F000F0, HM = 0x01000100), exactly.
template <uint32_t LO, uint32_t HM>
__device__ __forceinline__ uint32_t q5_f16x2(uint32_t lo, uint32_t hi)
{
    return (lo & LO) | (hi & HM) | 0x64006400u;
}

// int8 byte k of w (stored biased: byte ^ 0x80) as a float, exactly:
// 0x4B0000XX is 2^23 + XX.  (k is a constant once the caller's loop unrolls.)
__device__ __forceinline__ float sc_f32(uint32_t w_biased, int k)
{
    return __int_as_float((int)__byte_perm(w_biased, 0x4B000000u, 0x7540u | (uint32_t)k)) - 8388736.0f;
}

// One Q6_K job: superblock h of the chunk (8 blocks) in ring stage sq (ql box,
// then the qh box at 2048) and ss (sc box, then the superblock scales at 256)
// against staged blocks kb .. kb + 7.  Per block the two MMAs return the
// exact integer dots of the two 16-value halves, combined with the int8
// subscales (exact) and scaled by d_a in fp32; d6 once per job.
template <int M>
__device__ __forceinline__ void tc_job_q6_k(const uint8_t* sq, const uint8_t* ss, const uint8_t* act,
                                            const float* meta, int kb, int h, int g, int t,
                                            float (&acc)[(M + 7) / 8][4])
{
    constexpr int NT = (M + 7) / 8;
    float jacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) jacc[nt][i] = 0.0f;
    // ql: row g in line g (128-byte swizzle: piece p at p ^ (g & 7)), row g + 8
    // 1024 B on; qh: row g in line g of 64 B (64-byte swizzle: piece c at
    // c ^ ((g / 2) & 3)), row g + 8 512 B on
    const uint8_t* qlg = sq + g * 128 + 4 * t;
    const uint8_t* qhg = sq + 2048 + g * 64 + 4 * (t & 1);
    const int hsw = (g >> 1) & 3, sh = 4 - 4 * (t >> 1);
    const uint4 sva = *reinterpret_cast<const uint4*>(ss + g * 16);  // rows g, g + 8: sc of the 8 blocks
    const uint4 svb = *reinterpret_cast<const uint4*>(ss + (g + 8) * 16);
    const uint32_t sca[4] = {sva.x ^ 0x80808080u, sva.y ^ 0x80808080u, sva.z ^ 0x80808080u, sva.w ^ 0x80808080u};
    const uint32_t scb[4] = {svb.x ^ 0x80808080u, svb.y ^ 0x80808080u, svb.z ^ 0x80808080u, svb.w ^ 0x80808080u};
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const int swq = (p ^ g) << 4;
        const int hoff = (((p >> 1) ^ hsw) << 4) + (p & 1) * 8;
        const uint32_t wa = *reinterpret_cast<const uint32_t*>(qlg + swq);
        const uint32_t wb = *reinterpret_cast<const uint32_t*>(qlg + 1024 + swq);
        const uint32_t la = *reinterpret_cast<const uint32_t*>(qhg + hoff) << sh;
        const uint32_t lb = *reinterpret_cast<const uint32_t*>(qhg + 512 + hoff) << sh;
        // values (4t, 4t + 2) of rows g, g + 8, then (4t + 1, 4t + 3); the
        // same for the second half
        const uint32_t A0[4] = {q6_lo_f16x2(wa), q6_lo_f16x2(wb), q6_lo_f16x2(wa >> 8), q6_lo_f16x2(wb >> 8)};
        const uint32_t A1[4] = {q6_hi_f16x2(wa << 2, la), q6_hi_f16x2(wb << 2, lb), q6_hi_f16x2(wa >> 6, la >> 8),
                                q6_hi_f16x2(wb >> 6, lb >> 8)};
        // subscales of halves 0 and 1 of block p: bytes 2p, 2p + 1 of the row's 16
        const float s0a = sc_f32(sca[p >> 1], 2 * (p & 1)), s1a = sc_f32(sca[p >> 1], 2 * (p & 1) + 1);
        const float s0b = sc_f32(scb[p >> 1], 2 * (p & 1)), s1b = sc_f32(scb[p >> 1], 2 * (p & 1) + 1);
        const int b = kb + p;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int n = nt * 8 + g < M ? nt * 8 + g : M - 1;  // rows past M: any staged row (unused)
            const uint4 B = *reinterpret_cast<const uint4*>(act + (((size_t)b * M + n) * 4 + t) * 16);
            const float* mp = meta + (((size_t)b * NT + nt) * 4 + t) * 8;
            const float4 md = *reinterpret_cast<const float4*>(mp);
            const float2 mc = *reinterpret_cast<const float2*>(mp + 4);
            float d0[4], d1[4];
            mma_f16_16816(d0, A0, B.x, B.y, md.z, md.w, md.z, md.w);
            mma_f16_16816(d1, A1, B.z, B.w, mc.x, mc.y, mc.x, mc.y);
            // J = sc0 I0 + sc1 I1 (exact), then jacc += d_a J, in column pairs
            float ja0, ja1, jb0, jb1;
            mul_f32x2(ja0, ja1, s0a, s0a, d0[0], d0[1]);
            mul_f32x2(jb0, jb1, s0b, s0b, d0[2], d0[3]);
            fma_f32x2(ja0, ja1, s1a, s1a, d1[0], d1[1]);
            fma_f32x2(jb0, jb1, s1b, s1b, d1[2], d1[3]);
            fma_f32x2(jacc[nt][0], jacc[nt][1], md.x, md.y, ja0, ja1);
            fma_f32x2(jacc[nt][2], jacc[nt][3], md.x, md.y, jb0, jb1);
        }
    }
    // superblock scales of rows g, g + 8: group g / 4, row g % 4, superblock h
    const uint8_t* dp = ss + 256 + (g >> 2) * 32 + (g & 3) * 8 + h * 2;
    const float da6 = __half2float(*reinterpret_cast<const __half*>(dp));
    const float db6 = __half2float(*reinterpret_cast<const __half*>(dp + 64));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        acc[nt][0] = fmaf(da6, jacc[nt][0], acc[nt][0]);
        acc[nt][1] = fmaf(da6, jacc[nt][1], acc[nt][1]);
        acc[nt][2] = fmaf(db6, jacc[nt][2], acc[nt][2]);
        acc[nt][3] = fmaf(db6, jacc[nt][3], acc[nt][3]);
    }
}

// ---------------------------------------------------------------------------
// Q4_K: value d sc_b q - dmin m_b per 32-value block b.  The codes are in the
// Q4_0 nibble order, so the A registers and the staged activation are those
// of Q4_0 (no -8 offset: the start is C = -1024 sum lo - 64 sum hi); the
// scale and min terms in fp32: y += (d sc_b d_a) I_b - (dmin m_b) (d_a A_b).
// ---------------------------------------------------------------------------

// f * (unsigned byte k of w), exactly when the product fits fp32: the float
// with bits 0x4B0000XX is 2^23 + XX, and one fma of f with it against
// f_neg23 = -f * 2^23 leaves f * XX rounded once.
__device__ __forceinline__ float mul_u8(float f, float f_neg23, uint32_t w, int k)
{
    return fmaf(f, __int_as_float((int)__byte_perm(w, 0x4B000000u, 0x7540u | (uint32_t)k)), f_neg23);
}

// FIVE: Q5_K, whose fifth code bits (the word of row g, shifted right by t:
// byte k bit 0 = value 4t + k, bit 4 = value 16 + 4t + k) go to bit 4 (16 in
// the code 1024 + q) or bit 8 (16 in 1024 + 16 q) of each f16.
template <int M, bool FIVE>
__device__ __forceinline__ void tc_job_q4_k(const uint8_t* sn, const uint8_t* act, const float* meta, int kb, int g,
                                            int t, float (&acc)[(M + 7) / 8][4])
{
    constexpr int NT = (M + 7) / 8;
    constexpr int SCM = 8 * 256 + (FIVE ? 8 * TC_ROWS * 4 : 0);  // the {scale, min} bytes
    const uint8_t* codes = sn + (g * 4 + t) * 8;
    // rows g, g + 8: {scale, min} of the 8 blocks (16 B each), {d, dmin}
    const uint4 sma = *reinterpret_cast<const uint4*>(sn + SCM + g * 16);
    const uint4 smb = *reinterpret_cast<const uint4*>(sn + SCM + (g + 8) * 16);
    const uint32_t sa[4] = {sma.x, sma.y, sma.z, sma.w}, sb[4] = {smb.x, smb.y, smb.z, smb.w};
    const uint32_t dda = *reinterpret_cast<const uint32_t*>(sn + SCM + 8 * TC_ROWS * 2 + g * 4);
    const uint32_t ddb = *reinterpret_cast<const uint32_t*>(sn + SCM + 8 * TC_ROWS * 2 + (g + 8) * 4);
    const float da_w = __half2float(__ushort_as_half((unsigned short)(dda & 0xFFFFu)));
    const float dma_w = __half2float(__ushort_as_half((unsigned short)(dda >> 16)));
    const float db_w = __half2float(__ushort_as_half((unsigned short)(ddb & 0xFFFFu)));
    const float dmb_w = __half2float(__ushort_as_half((unsigned short)(ddb >> 16)));
    const float da_n = -8388608.0f * da_w, dma_n = -8388608.0f * dma_w;  // exact
    const float db_n = -8388608.0f * db_w, dmb_n = -8388608.0f * dmb_w;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const uint2 w = *reinterpret_cast<const uint2*>(codes + p * 256);
        const uint32_t wa8 = w.x >> 8, wb8 = w.y >> 8;
        uint32_t A0[4], A1[4];
        if constexpr (FIVE) {
            const uint32_t ha = *reinterpret_cast<const uint32_t*>(sn + 8 * 256 + (p * TC_ROWS + g) * 4) >> t;
            const uint32_t hb = *reinterpret_cast<const uint32_t*>(sn + 8 * 256 + (p * TC_ROWS + g + 8) * 4) >> t;
            const uint32_t ha4 = ha << 4, hb4 = hb << 4, ha_4 = ha >> 4, hb_4 = hb >> 4;
            A0[0] = q5_f16x2<0x000F000Fu, 0x00100010u>(w.x, ha4);
            A0[1] = q5_f16x2<0x000F000Fu, 0x00100010u>(w.y, hb4);
            A0[2] = q5_f16x2<0x000F000Fu, 0x00100010u>(wa8, ha_4);
            A0[3] = q5_f16x2<0x000F000Fu, 0x00100010u>(wb8, hb_4);
            A1[0] = q5_f16x2<0x00F000F0u, 0x01000100u>(w.x, ha4);
            A1[1] = q5_f16x2<0x00F000F0u, 0x01000100u>(w.y, hb4);
            A1[2] = q5_f16x2<0x00F000F0u, 0x01000100u>(wa8, ha_4);
            A1[3] = q5_f16x2<0x00F000F0u, 0x01000100u>(wb8, hb_4);
        } else {
            A0[0] = nib_f16x2<0x000F000Fu>(w.x);
            A0[1] = nib_f16x2<0x000F000Fu>(w.y);
            A0[2] = nib_f16x2<0x000F000Fu>(wa8);
            A0[3] = nib_f16x2<0x000F000Fu>(wb8);
            A1[0] = nib_f16x2<0x00F000F0u>(w.x);
            A1[1] = nib_f16x2<0x00F000F0u>(w.y);
            A1[2] = nib_f16x2<0x00F000F0u>(wa8);
            A1[3] = nib_f16x2<0x00F000F0u>(wb8);
        }
        // d sc and dmin m of block p, exact (fp16 x 6 bits): bytes 2 (p & 1),
        // + 1 of word p / 2
        const int k = 2 * (p & 1);
        const float Da = mul_u8(da_w, da_n, sa[p >> 1], k), Ma = mul_u8(dma_w, dma_n, sa[p >> 1], k + 1);
        const float Db = mul_u8(db_w, db_n, sb[p >> 1], k), Mb = mul_u8(dmb_w, dmb_n, sb[p >> 1], k + 1);
        const int b = kb + p;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int n = nt * 8 + g < M ? nt * 8 + g : M - 1;  // rows past M: any staged row (unused)
            const uint4 B = *reinterpret_cast<const uint4*>(act + (((size_t)b * M + n) * 4 + t) * 16);
            const float* mp = meta + ((size_t)b * NT + nt) * 24 + 2 * t;
            const float2 mda = *reinterpret_cast<const float2*>(mp);
            const float2 mc = *reinterpret_cast<const float2*>(mp + 8);
            const float2 me = *reinterpret_cast<const float2*>(mp + 16);
            float d[4];
            mma_f16_16816(d, A0, B.x, B.y, mc.x, mc.y, mc.x, mc.y);
            mma_f16_16816(d, A1, B.z, B.w, d[0], d[1], d[2], d[3]);
            float sa0, sa1, sb0, sb1;
            mul_f32x2(sa0, sa1, Da, Da, mda.x, mda.y);
            mul_f32x2(sb0, sb1, Db, Db, mda.x, mda.y);
            fma_f32x2(acc[nt][0], acc[nt][1], sa0, sa1, d[0], d[1]);
            fma_f32x2(acc[nt][2], acc[nt][3], sb0, sb1, d[2], d[3]);
            fma_f32x2(acc[nt][0], acc[nt][1], -Ma, -Ma, me.x, me.y);
            fma_f32x2(acc[nt][2], acc[nt][3], -Mb, -Mb, me.x, me.y);
        }
    }
}

// ---------------------------------------------------------------------------
// Q8_0 (fp16 d, int8 q[32], value d * q).  Its pack (qpack_q8_0) is built for
// this kernel: per 16-row tile, per job of 8 blocks one contiguous 4352-byte
// region = codes [block p][lane l][16 B] then scales [block p][row r] fp16,
// where lane l = 4g + t holds, as q + 128, values
//   2t, 2t+1, 2t+8, 2t+9, 16+2t, 17+2t, 24+2t, 25+2t
// of row g (bytes 0..7) and of row g + 8 (bytes 8..15): exactly its A
// fragments of the block's two m16n8k16 steps in natural K order, so one
// 16-byte load and one byte permute + one f16 subtract per register build them.
// The activation is staged in the same natural order, the accumulator starts
// at 0, and the block dot sum q_w q_a is exact (|partial sums| < 2^19).
// ---------------------------------------------------------------------------

// Bytes 0, 1 (sel 0x4140) or 2, 3 (sel 0x4342) of a word of biased codes
// (q + 128) as the f16x2 (q, q'), exactly: 0x6400 | (q + 128) is 1152 + q.
template <uint32_t SEL>
__device__ __forceinline__ uint32_t q8u_f16x2(uint32_t w)
{
    const uint32_t b = __byte_perm(w, 0x64646464u, SEL);
    const __half2 h = *reinterpret_cast<const __half2*>(&b);
    const __half2 r = __hsub2(h, __float2half2_rn(1152.0f));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// The activation for Q8_0: B fragments in natural K order, lane t of (block
// b, row n): (x[2t], x[2t+1]), (x[2t+8], x[2t+9]), (x[16+2t], ..), (x[24+2t], ..);
// meta {d_a, d_a', 0, 0}.  Same items and two phases as tc_stage_act.
template <int M>
__device__ __forceinline__ void tc_stage_act_q8_0(uint8_t* act, float* meta, const uint8_t* raw, int nkb, int rstride)
{
    constexpr int NT = (M + 7) / 8;
    constexpr int IT = 4 * tc_stage_items(M);
    const int total = nkb * NT * 32;
    uint32_t w0[IT], w1[IT];  // the lane's four code pairs, two per word
#pragma unroll
    for (int u = 0; u < IT; ++u) {
        const int i = threadIdx.x + u * TC_THREADS;
        w0[u] = w1[u] = 0;
        if (i >= total) break;
        const int tt = i & 3, n = ((i >> 5) % NT) * 8 + ((i >> 2) & 7), b = (i >> 5) / NT;
        float da = 0.0f;
        if (n < M) {
            const uint8_t* q = raw + (size_t)n * rstride + (size_t)b * Q8_1_BYTES + 4 + 2 * tt;
            const uint32_t p0 = *reinterpret_cast<const uint16_t*>(q), p1 = *reinterpret_cast<const uint16_t*>(q + 8);
            const uint32_t p2 = *reinterpret_cast<const uint16_t*>(q + 16), p3 = *reinterpret_cast<const uint16_t*>(q + 24);
            w0[u] = (p0 | p1 << 16) ^ 0x80808080u;
            w1[u] = (p2 | p3 << 16) ^ 0x80808080u;
            if (tt == 0) da = __half2float(*reinterpret_cast<const __half*>(q - 4));
        }
        if (tt == 0) {
            const int nt = n >> 3, c = n & 7;
            float* mp = meta + (((size_t)b * NT + nt) * 4 + (c >> 1)) * 4;
            mp[c & 1] = da;
            mp[2 + (c & 1)] = 0.0f;
        }
    }
    __syncthreads();  // the raw bytes are all read
#pragma unroll
    for (int u = 0; u < IT; ++u) {
        const int i = threadIdx.x + u * TC_THREADS;
        if (i >= total) break;
        const int tt = i & 3, n = ((i >> 5) % NT) * 8 + ((i >> 2) & 7), b = (i >> 5) / NT;
        if (n >= M) continue;
        uint4 v;
        v.x = q8u_f16x2<0x4140u>(w0[u]);
        v.y = q8u_f16x2<0x4342u>(w0[u]);
        v.z = q8u_f16x2<0x4140u>(w1[u]);
        v.w = q8u_f16x2<0x4342u>(w1[u]);
        *reinterpret_cast<uint4*>(act + (((size_t)b * M + n) * 4 + tt) * 16) = v;
    }
}

// One Q8_0 job: nblk (8, or 4 where shared memory is short) blocks in ring
// stage sn (their codes, then their scales at nblk * 512) against staged
// blocks kb .. kb + nblk - 1.
template <int M>
__device__ __forceinline__ void tc_job_q8_0(const uint8_t* sn, const uint8_t* act, const float* meta, int kb, int nblk,
                                            int g, int t, float (&acc)[(M + 7) / 8][4])
{
    constexpr int NT = (M + 7) / 8;
    float jacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) jacc[nt][i] = 0.0f;
    const uint8_t* codes = sn + (g * 4 + t) * 16;
    const uint8_t* dg = sn + nblk * 512 + g * 2;  // row g's scale; row g + 8's is 16 B on
#pragma unroll 1
    for (int p0 = 0; p0 < nblk; p0 += 4)
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
        const int p = p0 + pp;
        const uint4 w = *reinterpret_cast<const uint4*>(codes + p * 32 * 16);
        const float dwa = __half2float(*reinterpret_cast<const __half*>(dg + p * 32));
        const float dwb = __half2float(*reinterpret_cast<const __half*>(dg + p * 32 + 16));
        const uint32_t A0[4] = {q8u_f16x2<0x4140u>(w.x), q8u_f16x2<0x4140u>(w.z), q8u_f16x2<0x4342u>(w.x),
                                q8u_f16x2<0x4342u>(w.z)};
        const uint32_t A1[4] = {q8u_f16x2<0x4140u>(w.y), q8u_f16x2<0x4140u>(w.w), q8u_f16x2<0x4342u>(w.y),
                                q8u_f16x2<0x4342u>(w.w)};
        const int b = kb + p;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int n = nt * 8 + g < M ? nt * 8 + g : M - 1;
            const uint4 B = *reinterpret_cast<const uint4*>(act + (((size_t)b * M + n) * 4 + t) * 16);
            const float4 md = *reinterpret_cast<const float4*>(meta + (((size_t)b * NT + nt) * 4 + t) * 4);
            float d[4];
            mma_f16_16816(d, A0, B.x, B.y, 0.0f, 0.0f, 0.0f, 0.0f);
            mma_f16_16816(d, A1, B.z, B.w, d[0], d[1], d[2], d[3]);
            float sa0, sa1, sb0, sb1;
            mul_f32x2(sa0, sa1, dwa, dwa, md.x, md.y);
            mul_f32x2(sb0, sb1, dwb, dwb, md.x, md.y);
            fma_f32x2(jacc[nt][0], jacc[nt][1], sa0, sa1, d[0], d[1]);
            fma_f32x2(jacc[nt][2], jacc[nt][3], sb0, sb1, d[2], d[3]);
        }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] += jacc[nt][i];
}

// Write one tile's values, given as value index v of the fragment layout
// (lane = v / (4 NT), nt, i), to y.
template <int M>
__device__ __forceinline__ void tc_store(const TcArgs& a, int64_t T1, int64_t tau, int v, float val)
{
    constexpr int NT = (M + 7) / 8;
    const int ln = v / (4 * NT), rem = v - ln * (4 * NT), nt = rem >> 2, i = rem & 3;
    const int m = nt * 8 + 2 * (ln & 3) + (i & 1);
    if (m >= M) return;
    const bool second = tau >= T1;
    const int64_t n = (second ? tau - T1 : tau) * TC_ROWS + (ln >> 2) + (i >> 1) * 8;
    if (n >= (second ? a.N2 : a.N)) return;  // rows padding the last tile
    (second ? a.y2 : a.y)[(int64_t)m * a.ldy + n] = a.res ? val + a.res[(int64_t)m * a.ldr + n] : val;
}

template <int FMT, int M, bool PAIR>
__global__ void __launch_bounds__(TC_THREADS, 1)
    mmvq_tc_kernel(const TcArgs a, const __grid_constant__ CUtensorMap tn0, const __grid_constant__ CUtensorMap td0,
                        const __grid_constant__ CUtensorMap tn1, const __grid_constant__ CUtensorMap td1,
                        unsigned int* timeouts)
{
    constexpr int NT = (M + 7) / 8;
    constexpr int VT = 32 * NT * 4;  // values per tile
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr int W = TC_THREADS / 32;  // launched with exactly TC_THREADS threads
    const int lane = threadIdx.x & 31;
    const int warp = __shfl_sync(FULL, (int)(threadIdx.x >> 5), 0);
    const int g = lane >> 2, t = lane & 3;
    const int S = a.stages;
    pdl_launch_dependents();

    // This CTA's tiles (its cluster's) and K part (its rank's).  The special
    // registers are broadcast so that everything derived from them, down to
    // the copy coordinates, is warp-uniform.
    const int C = __shfl_sync(FULL, (int)cluster_nctarank(), 0);
    const int rank = __shfl_sync(FULL, (int)cluster_ctarank(), 0);
    const int ncl = __shfl_sync(FULL, (int)cluster_count_x(), 0);
    const int cl = __shfl_sync(FULL, (int)cluster_id_x(), 0);
    const int NB = a.K / QK;
    const int T1 = (a.N + TC_ROWS - 1) / TC_ROWS, T = T1 + (PAIR ? (a.N2 + TC_ROWS - 1) / TC_ROWS : 0);
    // (32-bit divisions where the products fit)
    const bool narrow = (int64_t)ncl * T <= (int64_t)0xFFFFFFFFu;
    const int t0 = narrow ? (int)((uint32_t)cl * (uint32_t)T / (uint32_t)ncl) : (int)((int64_t)cl * T / ncl);
    const int t1 = narrow ? (int)((uint32_t)(cl + 1) * (uint32_t)T / (uint32_t)ncl) : (int)((int64_t)(cl + 1) * T / ncl);
    const int ntile = t1 - t0;
    const int JB = a.jb;
    const int NIB = FMT == TCF_Q8_0   ? tc_q8_0_job_bytes(JB)
                    : FMT == TCF_Q6_K ? TC_Q6_K_NIB
                    : FMT == TCF_Q4_K ? TC_Q4_K_JOB * (JB / 8)
                    : FMT == TCF_Q5_K ? TC_Q5_K_JOB * (JB / 8)
                                      : tc_nib_bytes(JB);
    const int DSB = FMT == TCF_Q6_K ? TC_Q6_K_DS : FMT == TCF_Q4_0 ? tc_ds_bytes(JB) : 0;
    const int JPC = CHUNK / JB, JPC_LOG = JB > TC_LINE_JB ? 1 : 2;  // jobs per 32-block chunk
    const int njb = NB / JB;
    const int jb0 = rank * njb / C, jb1 = (rank + 1) * njb / C;
    const int jpt = jb1 - jb0;  // jobs per tile
    const int J = ntile * jpt;
    const int j0 = warp * J / W, j1 = (warp + 1) * J / W;
    const TcSmem sl = tc_smem(M, W, S, a.nkb_max, C > 1 ? a.out_tiles : 0, NIB, DSB,
                              tc_meta_bytes(FMT));
    // (debug build: the layout must fit the launch's shared memory; every CTA
    // of a cluster decides alike, so none waits on a CTA that left)
    if (!QG_OK(sl.bytes <= dynamic_smem_bytes(), timeouts, 810)) return;
    uint8_t* nib = smem + sl.nib;
    uint8_t* ds = smem + sl.ds;
    uint8_t* act = smem + sl.act;
    float* meta = reinterpret_cast<float*>(smem + sl.meta);
    float* outb = reinterpret_cast<float*>(smem + sl.out);
    int* tab = reinterpret_cast<int*>(smem + sl.tab);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + sl.bar);
    uint64_t* wbar = bars + warp * S;
    uint64_t* abar = bars + W * S;  // the activation copy
    uint8_t* wnib = nib + (size_t)warp * S * NIB;
    uint8_t* wds = ds + (size_t)warp * S * DSB;

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&wbar[s], 1);
        if (warp == 0) mbar_init(abar, 1);
        fence_barrier_init();
    }
    if ((FMT == TCF_Q4_0 || FMT == TCF_Q6_K) && warp == 1 && lane < (PAIR || FMT == TCF_Q6_K ? 4 : 2)) {
        // bring the copies' descriptors on chip while the prologue runs
        const CUtensorMap* map = lane == 0 ? &tn0 : lane == 1 ? &td0 : lane == 2 ? &tn1 : &td1;
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
    }
    __syncthreads();  // barriers initialized
    const uint64_t pol = __shfl_sync(FULL, l2_evict_first_policy(), 0);  // warp-uniform copy operand

    // The consumer walks the jobs as (CTA-local tile, job within the tile);
    // the copy issue keeps its own running coordinates.
    struct Cursor {
        int tau, kj;
    };
    auto start = [&](int j) {
        Cursor c;
        c.tau = jpt > 0 ? j / jpt : 0;
        c.kj = j - c.tau * jpt;
        return c;
    };
    int issued = 0, iss_slot = 0;
    const int n_jobs = j1 - j0;
    // next copy: job ikj of the tile whose first group is igrp (of the
    // second weight when isec), blocks 8 ikg .. 8 ikg + 7 of the row
    int ikj, ikg, igrp;
    bool isec;
    {
        const Cursor c = start(j0);
        const int tg = t0 + c.tau;
        ikj = c.kj;
        ikg = jb0 + c.kj;
        isec = PAIR && tg >= T1;
        igrp = (isec ? tg - T1 : tg) * (TC_ROWS / GROUP);
    }
    auto issue = [&]() {
        const int h = ikg & (JPC - 1), c = ikg >> JPC_LOG;  // which JB blocks of which 32-block chunk
        // (debug build: a job outside its weight completes its stage empty)
        const int Nw = isec ? a.N2 : a.N;
        const int64_t T16 = (Nw + TC_ROWS - 1) / TC_ROWS;
        const int PER = JB < TC_Q8_0_JOB_BLOCKS ? TC_Q8_0_JOB_BLOCKS / JB : 1;  // Q8_0 jobs per region
        const bool ok = QG_OK(FMT == TCF_Q8_0   ? qg_in(((int64_t)(igrp >> 2) * (njb / PER) + ikg / PER) * TC_Q8_0_JOB,
                                                       TC_Q8_0_JOB, T16 * (njb / PER) * TC_Q8_0_JOB)
                              : (FMT == TCF_Q4_K || FMT == TCF_Q5_K)
                                  ? qg_in(((int64_t)(igrp >> 2) * njb + ikg) * NIB, NIB, T16 * njb * NIB)
                                  : igrp >= 0 && igrp < Nw / GROUP && c < (NB + CHUNK - 1) / CHUNK,
                              timeouts, 801);
        if (lane == 0) {
            uint64_t* bar = &wbar[iss_slot];
            uint8_t* dst = wnib + (size_t)iss_slot * NIB;
            fence_proxy_async();
            mbar_arrive_expect_tx(bar, ok ? NIB + DSB : 0u);
            if (!ok) {
            } else if constexpr (FMT == TCF_Q8_0) {
                // the job's part of the Q8_0 pack: tile igrp / 4, region (8
                // blocks) ikg * JB / 8, all of it or the half h of its codes
                // and of its scales
                const int per = TC_Q8_0_JOB_BLOCKS / JB, reg = ikg / per, hh = ikg - reg * per;
                const uint8_t* src = (isec ? a.w1 : a.w0) +
                                     ((int64_t)(igrp >> 2) * (njb / per) + reg) * TC_Q8_0_JOB;
                if (per == 1) {
                    bulk_g2s(dst, src, TC_Q8_0_JOB, bar, pol);
                } else {
                    bulk_g2s(dst, src + hh * JB * 512, JB * 512, bar, pol);
                    bulk_g2s(dst + JB * 512, src + TC_Q8_0_CODES + hh * JB * 32, JB * 32, bar, pol);
                }
            } else if constexpr (FMT == TCF_Q4_K || FMT == TCF_Q5_K) {
                // the job's JB / 8 regions of the pack (adjacent): tile igrp / 4,
                // superblocks ikg * JB / 8 ..
                bulk_g2s(dst, a.w0 + ((int64_t)(igrp >> 2) * njb + ikg) * NIB, NIB, bar, pol);
            } else if constexpr (FMT == TCF_Q6_K) {
                // superblock h of chunk c for the tile's 16 rows: ql, qh and sc
                // boxes of the row tiles, then the chunk's superblock scales
                uint8_t* ds = wds + (size_t)iss_slot * DSB;
                tma_load_4d(dst, &tn0, h * 128, 0, c, igrp, bar, pol);
                tma_load_4d(dst + TC_ROWS * 128, &td0, CHUNK * 16 + h * 64, 0, c, igrp, bar, pol);
                tma_load_4d(ds, &tn1, CHUNK * 24 + h * 16, 0, c, igrp, bar, pol);
                tma_load_3d(ds + TC_ROWS * 16, &td1, 0, c, igrp, bar, pol);
            } else {
                const CUtensorMap* map = isec ? &tn1 : &tn0;
                tma_load_4d(dst, map, h * JB * 16, 0, c, igrp, bar, pol);
                if (JB > TC_LINE_JB) tma_load_4d(dst + TC_BOX, map, h * JB * 16 + 128, 0, c, igrp, bar, pol);
                tma_load_3d(wds + (size_t)iss_slot * DSB, isec ? &td1 : &td0, h * JB * 8, c, igrp, bar, pol);
            }
        }
        ++ikg;
        if (++ikj == jpt) {  // next tile
            ikj = 0;
            ikg = jb0;
            igrp += TC_ROWS / GROUP;
            if (PAIR && !isec && igrp == T1 * (TC_ROWS / GROUP)) {
                isec = true;
                igrp = 0;
            }
        }
        ++issued;
        if (++iss_slot == S) iss_slot = 0;
    };
    pdl_wait();

    // The activation's K part: one bulk copy per row into the tail of the
    // tile region; the ring starts at once (every earlier kernel's writes are
    // visible from here) and fills while the copy is converted.
    bool alive = true;
    const uint32_t row_bytes = (uint32_t)jpt * JB * Q8_1_BYTES, rstride = row_bytes + 16;
    uint8_t* raw = act + (size_t)a.nkb_max * M * 64 - (size_t)M * rstride;
    if (threadIdx.x == 0 && row_bytes > 0) {
        const bool ok = QG_OK(qg_in(((int64_t)(M - 1) * NB + (int64_t)jb0 * JB) * Q8_1_BYTES, row_bytes,
                                    (int64_t)M * NB * Q8_1_BYTES),
                              timeouts, 802);
        mbar_arrive_expect_tx(abar, ok ? (uint32_t)M * row_bytes : 0u);
        for (int n = 0; ok && n < M; ++n)
            bulk_g2s_plain(raw + (size_t)n * rstride, a.xq + ((int64_t)n * NB + (int64_t)jb0 * JB) * Q8_1_BYTES,
                           row_bytes, abar);
    }
    while (issued < n_jobs && issued < S - 1) issue();
    if (warp == W - 1) {  // while the activation copy is in flight
        // Tiles cut by a warp boundary (found at the first boundary strictly
        // inside them): the tile, the warps holding its pieces (a mask), and
        // whether the first of them holds it in its second slot.
        const int w = lane + 1;
        bool split = false;
        int tau = 0, mask = 0, sa = 0;
        if (w < W && jpt > 0) {
            const int bnd = w * J / W, prev = (w - 1) * J / W;
            tau = bnd / jpt;
            split = bnd % jpt != 0 && prev <= tau * jpt;
            if (split) {
                const int first = tau * jpt, last = first + jpt - 1;
                const int wa = ((first + 1) * W - 1) / J, wb = ((last + 1) * W - 1) / J;
                for (int ww = wa; ww <= wb; ++ww)
                    if (ww * J / W != (ww + 1) * J / W) mask |= 1 << ww;  // skip empty warps
                sa = wa * J / W < first ? 1 : 0;
            }
        }
        const unsigned sel = __ballot_sync(FULL, split);
        if (split) {
            const int e = __popc(sel & ((1u << lane) - 1));
            tab[1 + 3 * e] = tau;
            tab[2 + 3 * e] = mask;
            tab[3 + 3 * e] = sa;
        }
        if (lane == 0) tab[0] = __popc(sel);
    }

    if (row_bytes > 0 && !__all_sync(FULL, mbar_wait_bounded(abar, 0))) {
        if (lane == 0) atomicAdd_system(timeouts, 1u);
        alive = false;
    }
    alive = __syncthreads_and(alive);
    if (alive) {
        if constexpr (FMT == TCF_Q8_0) tc_stage_act_q8_0<M>(act, meta, raw, jpt * JB, (int)rstride);
        else tc_stage_act<M, FMT>(act, meta, raw, jpt * JB, (int)rstride);
    }
    __syncthreads();  // the tile is built
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
    // A warp's pieces of cut tiles (its first segment, its last) wait in
    // registers until the loop ends; they go to the ring area afterwards.
    float first_piece[NT][4];
    bool has_first = false, has_last = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) first_piece[nt][i] = 0.0f;
    int slot = 0, consumed = 0, seg_begin = j0;
    uint32_t phase = 0;
    const Cursor first = start(j0);
    int tl = first.tau, kj = first.kj;  // the job being worked on: tile (CTA-local) and job within it
    for (int j = j0; alive && j < j1; ++j) {
        if (issued < n_jobs) issue();
        if (!__all_sync(FULL, mbar_wait_bounded(&wbar[slot], phase))) {
            if (lane == 0) atomicAdd_system(timeouts, 1u);
            break;
        }
        ++consumed;
        if constexpr (FMT == TCF_Q8_0) tc_job_q8_0<M>(wnib + (size_t)slot * NIB, act, meta, kj * JB, JB, g, t, acc);
        else if constexpr (FMT == TCF_Q4_K || FMT == TCF_Q5_K) {
            constexpr int RB = FMT == TCF_Q5_K ? TC_Q5_K_JOB : TC_Q4_K_JOB;
#pragma unroll 1
            for (int r = 0; r < JB / 8; ++r)  // one superblock region at a time
                tc_job_q4_k<M, FMT == TCF_Q5_K>(wnib + (size_t)slot * NIB + r * RB, act, meta, kj * JB + 8 * r, g, t,
                                                acc);
        }
        else if constexpr (FMT == TCF_Q6_K)
            tc_job_q6_k<M>(wnib + (size_t)slot * NIB, wds + (size_t)slot * DSB, act, meta, kj * JB,
                           (jb0 + kj) & (JPC - 1), g, t, acc);
        else tc_job<M>(wnib + (size_t)slot * NIB, wds + (size_t)slot * DSB, act, meta, kj * JB, JB, g, t, acc);
        __syncwarp();
        if (++slot == S) {
            slot = 0;
            phase ^= 1u;
        }
        const bool tile_end = ++kj == jpt;
        if (tile_end || j + 1 == j1) {
            // a segment of tile tl ends: whole tiles go out; a piece of a cut
            // tile is the warp's first segment (kept) or its last (left in acc)
            const bool whole = tile_end && seg_begin == tl * jpt;
            if (whole || seg_begin == j0) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (!whole) first_piece[nt][i] = acc[nt][i];
                        else if (C > 1) outb[(size_t)tl * VT + lane * NT * 4 + nt * 4 + i] = acc[nt][i];
                        else tc_store<M>(a, T1, t0 + tl, lane * NT * 4 + nt * 4 + i, acc[nt][i]);
                        acc[nt][i] = 0.0f;
                    }
                has_first = has_first || !whole;
            } else {
                has_last = true;  // ends at j1: the loop ends with it
            }
            seg_begin = j + 1;
            if (tile_end) {
                ++tl;
                kj = 0;
            }
        }
    }
    // After a timeout, give the copies still in flight a bounded wait before
    // the shared memory is released.
    if (lane == 0) {
        for (int jj = consumed; jj < issued; ++jj) mbar_wait_bounded(&wbar[jj % S], (uint32_t)((jj / S) & 1));
        if (!alive && warp == 0) mbar_wait_bounded(abar, 0);
    }
    __syncthreads();  // the ring area is free
    float* slots = reinterpret_cast<float*>(nib);  // [warp][first, last][lane] x 4 NT floats
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (has_first) slots[((size_t)(warp * 2) * 32 + lane) * NT * 4 + nt * 4 + i] = first_piece[nt][i];
            if (has_last) slots[((size_t)(warp * 2 + 1) * 32 + lane) * NT * 4 + nt * 4 + i] = acc[nt][i];
        }
    __syncthreads();

    // Tiles cut by a warp boundary: their pieces added in warp order.
    const int ne = tab[0];
    for (int o = threadIdx.x; o < ne * VT; o += blockDim.x) {
        const int e = o / VT, v = o - e * VT;
        const int tau = tab[1 + 3 * e];
        unsigned mask = (unsigned)tab[2 + 3 * e];
        const int wa = __ffs(mask) - 1;
        float sum = slots[(size_t)(wa * 2 + tab[3 + 3 * e]) * VT + v];
        mask &= mask - 1;
        while (mask) {
            const int ww = __ffs(mask) - 1;
            mask &= mask - 1;
            sum += slots[(size_t)(ww * 2) * VT + v];
        }
        if (C > 1) outb[(size_t)tau * VT + v] = sum;
        else tc_store<M>(a, T1, t0 + tau, v, sum);
    }
    if (C > 1) {
        // The K parts of each tile, added in rank order; rank r writes its
        // share of the cluster's tiles.
        cluster_sync_all();
        const int ta = rank * ntile / C, tb = (rank + 1) * ntile / C;
        for (int o = threadIdx.x; o < (tb - ta) * VT; o += blockDim.x) {
            const int tau = ta + o / VT, v = o - (tau - ta) * VT;
            const float* p = outb + (size_t)tau * VT + v;
            float sum = ld_dsmem_f32(p, 0);
            for (int rr = 1; rr < C; ++rr) sum += ld_dsmem_f32(p, (uint32_t)rr);
            tc_store<M>(a, T1, t0 + tau, v, sum);
        }
        cluster_sync_all();  // no CTA leaves while its shared memory is read
    }
}

}  // namespace qgemv
