// Q4_0 x Q8_1 MMVQ for M <= 8 activation rows on the tensor cores: the form
// of the tensor-core kernel for a single 8-column MMA tile, written for the
// fewest instructions per weight block, which is what bounds the width-6
// verifier projections ("Qwen3.6 27B Q4_0 DFlash/SYCL closure", Objective and
// final result: the width-6 target MLP sets the cycle time; What materially
// worked, item 2: direct Q4_0 MMVQ).
//
// The arithmetic is exactly that of mmvq_tc_kernel (exact integer block dots
// from f16 mma.sync m16n8k16 with the accumulator started at
// -1032 sum_{i<16} q_a - 72 sum_{i>=16} q_a, then y += (d_w d_a) I in fp32,
// summed per job, then across jobs), on the same packed weight read through
// the same two TMA tensor maps.  What differs is how the work is issued:
//   * a job is a unit of TL 16-row tiles (one, or two sharing every load of
//     the activation's B fragments and meta, which halves the shared-memory
//     traffic per weight block that bounds the loop) times JB blocks (8 or
//     16), both compile-time constants; every shared-memory access uses a
//     32-bit address with a constant offset;
//   * one ldmatrix.x4 per two blocks gathers, for the lane (g, t), the code
//     words of rows g and g + 8 of both blocks out of the 128-byte-swizzled
//     code box (four LDS and their address arithmetic before);
//   * the activation's K part is bulk-copied first (it is on every job's
//     path), the ring copies after it; it is converted one (block, row) unit
//     per thread: eight dp4a give the two code sums, no shuffles, and the
//     records are written in a rotated order that keeps the 16-byte stores
//     free of bank conflicts;
//   * a job's copy is issued by its own warp right after the job before it in
//     the same ring stage is done, so S jobs are in flight during every wait
//     (one warp issuing every copy was slower: each tensor copy holds its
//     issuing thread for some hundred cycles).
// The CTA ranges (in units), the per-warp job ranges, the combine of units
// cut between warps (in warp order) and of K parts across a cluster (in rank
// order) are those of mmvq_tc_kernel: the result does not depend on timing.
#pragma once

#include "mmvq_tc.cuh"

namespace qgemv {

constexpr int QM_THREADS = 512;
constexpr int QM_WARPS = QM_THREADS / 32;
constexpr int QM_UNITS = 4;      // activation (block, row) units per thread, at most
constexpr int QM_MAX_STAGES = 8;
constexpr int QM_VT = 128;       // values of one 16-row tile's fragment: 32 lanes x 4

struct QmSmem {
    uint32_t nib, ds, act, meta, out, tab, bar, bytes;
};

// Shared-memory layout, identical on the host (sizing) and the device: ring
// stages of codes (1024-byte aligned: 128-byte swizzle atoms), of scales, the
// activation's B fragments [block][row][lane t] x 16 B, its meta per block
// ([lane t] x {C, C', C, C'}, the accumulator start as a ready register quad,
// then [lane t] x {d_a, d_a'}), the cluster combine area, the cut-unit table
// and the ring barriers.
// TL: 16-row tiles per unit (a job is TL tiles x JB blocks); out_units:
// the units of the cluster combine area.
__host__ __device__ inline QmSmem qm_smem(int M, int S, int JB, int TL, int nkb, int out_units)
{
    QmSmem s;
    uint32_t o = 0;
    s.nib = o;  o += (uint32_t)QM_WARPS * S * TL * JB * 256;
    s.ds = o;   o += (uint32_t)QM_WARPS * S * TL * JB * 32;
    s.act = o;  o += (uint32_t)nkb * M * 64;
    s.meta = o; o += (uint32_t)nkb * 96;
    s.out = o;  o += (uint32_t)out_units * TL * QM_VT * 4;
    s.tab = o;  o += TC_TAB_INTS * 4;
    s.bar = o;  o += (uint32_t)(QM_WARPS * S + 1) * 8;  // ring barriers, then the activation's
    s.bytes = o + 1024;  // room to align the base to 1024 B
    return s;
}

// ---------------------------------------------------------------------------
// 32-bit shared-memory accesses.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint4 lds_v4(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// An fp16 value in shared memory, widened to fp32 (exact).
__device__ __forceinline__ float lds_f16(uint32_t a)
{
    float f;
    asm volatile("{\n\t.reg .b16 h;\n\tld.shared.b16 h, [%1];\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "r"(a));
    return f;
}

__device__ __forceinline__ void sts_v4(uint32_t a, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void sts_u32(uint32_t a, uint32_t v)
{
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Four 8 x 8 matrices of 16-bit elements; lanes 8i .. 8i + 7 give the row
// addresses of matrix i, and lane 4 r + c receives elements 2c, 2c + 1 of row
// r of each matrix: bytes 4c .. 4c + 3 of the 16-byte row.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t a)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}

// ---------------------------------------------------------------------------
// Activation staging: the CTA's K part of the Q8_1 activation as the B
// fragments and meta that mmvq_tc_kernel stages (same values, same layout for
// one 8-row tile), one (block b, row n) unit per thread and round.
//   record (b, n, lane t): f16x2 (q[4t], q[4t+2]), (q[4t+1], q[4t+3]),
//                          (q[16+4t], q[16+4t+2]) / 16, (q[16+4t+1], q[16+4t+3]) / 16
//   meta (b): [lane t] {C[2t], C[2t+1], C[2t], C[2t+1]} (64 B), then [lane t]
//             {d_a[2t], d_a[2t+1]} (32 B); zero for rows >= M.
// Units are numbered n fastest, so a warp's 16-byte stores land on 32
// consecutive 64-byte records; unit u writes its four 16-byte pieces in the
// order (k + u / 2) mod 4, which puts the eight stores of each quarter-warp
// phase in distinct bank groups.
// ---------------------------------------------------------------------------
// Phase 1: the thread's units' Q8_1 bytes into registers, from the raw copy
// of the CTA's K part in shared memory (row n's blocks at raw + n rstride).
template <int M>
__device__ __forceinline__ void qm_stage_load(uint32_t (&w)[QM_UNITS][9], uint32_t raw, int rstride, int nkb)
{
    const int nunits = nkb * M;
#pragma unroll
    for (int u = 0; u < QM_UNITS; ++u) {
        const int i = threadIdx.x + u * QM_THREADS;
        if (i < nunits) {
            const int b = i / M, n = i - b * M;
            const uint32_t src = raw + (uint32_t)(n * rstride + b * Q8_1_BYTES);
#pragma unroll
            for (int k = 0; k < 9; ++k) asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w[u][k]) : "r"(src + 4 * k));
        }
    }
}

// Phase 2: the records and meta of the thread's units.
template <int M>
__device__ __forceinline__ void qm_stage_store(const uint32_t (&w)[QM_UNITS][9], uint32_t act, uint32_t meta, int nkb)
{
    const int nunits = nkb * M;
#pragma unroll
    for (int u = 0; u < QM_UNITS; ++u) {
        const int i = threadIdx.x + u * QM_THREADS;
        if (i >= nunits) break;
        const int b = i / M, n = i - b * M;
        int s_lo = 0, s_hi = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            s_lo = __dp4a((int)w[u][1 + k], 0x01010101, s_lo);
            s_hi = __dp4a((int)w[u][5 + k], 0x01010101, s_hi);
        }
        const uint32_t rec = act + (uint32_t)i * 64;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int k = (kk + (i >> 1)) & 3;
            uint32_t q0 = w[u][1], q1 = w[u][5];  // (k chosen at run time: pick the lane's words)
            q0 = k == 1 ? w[u][2] : k == 2 ? w[u][3] : k == 3 ? w[u][4] : q0;
            q1 = k == 1 ? w[u][6] : k == 2 ? w[u][7] : k == 3 ? w[u][8] : q1;
            uint4 v;
            v.x = q8_f16x2<0x4240u, false>(q0);
            v.y = q8_f16x2<0x4341u, false>(q0);
            v.z = q8_f16x2<0x4240u, true>(q1);
            v.w = q8_f16x2<0x4341u, true>(q1);
            sts_v4(rec + k * 16, v);
        }
        const float da = __half2float(__ushort_as_half((unsigned short)(w[u][0] & 0xFFFFu)));
        const uint32_t mp = meta + (uint32_t)b * 96 + (n >> 1) * 16 + (n & 1) * 4;
        const uint32_t cv = __float_as_uint((float)(-1032 * s_lo - 72 * s_hi));
        sts_u32(mp, cv);
        sts_u32(mp + 8, cv);
        sts_u32(meta + (uint32_t)b * 96 + 64 + (n >> 1) * 8 + (n & 1) * 4, __float_as_uint(da));
    }
    if constexpr (M < 8) {
        // rows M .. 7 of every block: zero scale and start
        constexpr int PAD = 8 - M;
        for (int i = threadIdx.x; i < nkb * PAD; i += QM_THREADS) {
            const int b = i / PAD, n = M + (i - b * PAD);
            const uint32_t mp = meta + (uint32_t)b * 96 + (n >> 1) * 16 + (n & 1) * 4;
            sts_u32(mp, 0u);
            sts_u32(mp + 8, 0u);
            sts_u32(meta + (uint32_t)b * 96 + 64 + (n >> 1) * 8 + (n & 1) * 4, 0u);
        }
    }
}

// ---------------------------------------------------------------------------
// One job: JB blocks of a unit of TL 16-row tiles.
//   sn: the lane's ldmatrix row address for blocks 0 and 1 of the stage's
//       first code box: line L = (lane & 7) + 8 ((lane >> 3) & 1) (rows g,
//       then g + 8), 16-byte piece c = ((lane >> 4) & 1) ^ (lane & 7) (blocks
//       p, then p + 1, under the swizzle); the box of tile u and blocks
//       8h .. 8h + 7 is 2048 (u JB / 8 + h) bytes on, and blocks p, p + 1 of
//       it are at (box + sn) ^ ((p mod 8) << 4), p even;
//   sd: the lane's scale of row g for block 0 of tile 0: [4 TL groups][JB
//       blocks][4 rows] fp16; row g + 8 two groups on, tile u 4u groups on;
//   bA: the B fragment (lane t) of block 0 of the job, row min(g, M - 1);
//   bM: the accumulator-start quad (lane t) of block 0 of the job; its d_a
//       pair is 64 - 8t bytes on.
// acc[u] (tile u: rows g, g, g + 8, g + 8; columns 2t, 2t + 1, 2t, 2t + 1)
// += the job's sum.  The activation fragment and meta of a block are loaded
// once for the TL tiles.
// ---------------------------------------------------------------------------
template <int M, int JB, int TL>
__device__ __forceinline__ void qm_job(uint32_t sn, uint32_t sd, uint32_t bA, uint32_t bM, float (&acc)[TL][4])
{
    const uint32_t bD = bM + 64 - (threadIdx.x & 3) * 8;  // the lane's d_a pairs
    float j[TL][4];
#pragma unroll
    for (int u = 0; u < TL; ++u)
#pragma unroll
        for (int i = 0; i < 4; ++i) j[u][i] = 0.0f;
#pragma unroll
    for (int p = 0; p < JB; p += 2) {
        uint32_t cw[TL][4];
#pragma unroll
        for (int u = 0; u < TL; ++u)
            ldsm_x4(cw[u], (sn + (uint32_t)(u * (JB / 8) + (p >> 3)) * 2048u) ^ ((uint32_t)(p & 7) << 4));
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int pb = p + q;
            const uint4 B = lds_v4(bA + pb * M * 64);
            const uint4 cq = lds_v4(bM + pb * 96);
            uint2 dd;
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(dd.x), "=r"(dd.y) : "r"(bD + pb * 96));
            const float da0 = __uint_as_float(dd.x), da1 = __uint_as_float(dd.y);
#pragma unroll
            for (int u = 0; u < TL; ++u) {
                const uint32_t wa = cw[u][2 * q], wb = cw[u][2 * q + 1];
                const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
                const uint32_t A0[4] = {nib_f16x2<0x000F000Fu>(wa), nib_f16x2<0x000F000Fu>(wb),
                                        nib_f16x2<0x000F000Fu>(wa8), nib_f16x2<0x000F000Fu>(wb8)};
                const uint32_t A1[4] = {nib_f16x2<0x00F000F0u>(wa), nib_f16x2<0x00F000F0u>(wb),
                                        nib_f16x2<0x00F000F0u>(wa8), nib_f16x2<0x00F000F0u>(wb8)};
                const float dwa = lds_f16(sd + u * (4 * JB * 8) + pb * 8);
                const float dwb = lds_f16(sd + u * (4 * JB * 8) + 2 * JB * 8 + pb * 8);
                float d[4];
                mma_f16_16816(d, A0, B.x, B.y, __uint_as_float(cq.x), __uint_as_float(cq.y), __uint_as_float(cq.z),
                              __uint_as_float(cq.w));
                mma_f16_16816(d, A1, B.z, B.w, d[0], d[1], d[2], d[3]);
                // j += (d_w d_a) I, the exact fp16 x fp16 product first
                float sa0, sa1, sb0, sb1;
                mul_f32x2(sa0, sa1, dwa, dwa, da0, da1);
                mul_f32x2(sb0, sb1, dwb, dwb, da0, da1);
                fma_f32x2(j[u][0], j[u][1], sa0, sa1, d[0], d[1]);
                fma_f32x2(j[u][2], j[u][3], sb0, sb1, d[2], d[3]);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < TL; ++u)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[u][i] += j[u][i];
}

// Write value v of a unit's fragments (tile v / 128, then the layout of
// tc_store) to y; units of the second weight (PAIR) follow the first's.
template <int M, int TL>
__device__ __forceinline__ void qm_store(const TcArgs& a, int U1, int unit, int v, float val)
{
    const int u = v >> 7, r = v & 127;
    const int ln = r >> 2, i = r & 3;
    const int m = 2 * (ln & 3) + (i & 1);
    if (m >= M) return;
    const bool second = unit >= U1;
    const int64_t n = ((int64_t)(second ? unit - U1 : unit) * TL + u) * TC_ROWS + (ln >> 2) + (i >> 1) * 8;
    if (n >= (second ? a.N2 : a.N)) return;  // rows padding the last unit
    (second ? a.y2 : a.y)[(int64_t)m * a.ldy + n] = a.res ? val + a.res[(int64_t)m * a.ldr + n] : val;
}

template <int M, int JB, int TL, bool PAIR>
__global__ void __launch_bounds__(QM_THREADS, 1)
    mmvq_q4_0_mma_kernel(const TcArgs a, const __grid_constant__ CUtensorMap tn0,
                         const __grid_constant__ CUtensorMap td0, const __grid_constant__ CUtensorMap tn1,
                         const __grid_constant__ CUtensorMap td1, unsigned int* timeouts)
{
    static_assert(M >= 1 && M <= 8, "one 8-column MMA tile");
    static_assert(JB == 8 || JB == 16, "8 or 16 blocks per job");
    static_assert(TL == 1 || (TL == 2 && JB == 8), "one tile per unit, or two with 8-block jobs");
    constexpr int W = QM_WARPS;
    constexpr int VU = TL * QM_VT;  // values of a unit's fragments
    constexpr int NIB = TL * JB * 256, DSB = TL * JB * 32;
    constexpr int JPC = CHUNK / JB, JPC_LOG = JB == 16 ? 1 : 2;  // jobs per 32-block chunk
    constexpr int UG = TL * TC_ROWS / GROUP;                      // 4-row groups per unit
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t s_raw = smem_u32(smem_raw);
    const uint32_t sb = (s_raw + 1023u) & ~1023u;  // 1024-aligned base (shared address)
    uint8_t* smem = smem_raw + (sb - s_raw);
    const int lane = threadIdx.x & 31;
    const int warp = __shfl_sync(FULL, (int)(threadIdx.x >> 5), 0);
    const int g = lane >> 2, t = lane & 3;
    const int S = a.stages;
    pdl_launch_dependents();

    // This CTA's units (its cluster's) and K part (its rank's), warp-uniform.
    const int C = __shfl_sync(FULL, (int)cluster_nctarank(), 0);
    const int rank = __shfl_sync(FULL, (int)cluster_ctarank(), 0);
    const int ncl = __shfl_sync(FULL, (int)cluster_count_x(), 0);
    const int cl = __shfl_sync(FULL, (int)cluster_id_x(), 0);
    const int NB = a.K / QK;
    const int U1 = (a.N / TC_ROWS + TL - 1) / TL, T = U1 + (PAIR ? (a.N2 / TC_ROWS + TL - 1) / TL : 0);
    const bool narrow = (int64_t)ncl * T <= (int64_t)0xFFFFFFFFu;
    const int t0 = narrow ? (int)((uint32_t)cl * (uint32_t)T / (uint32_t)ncl) : (int)((int64_t)cl * T / ncl);
    const int t1 =
        narrow ? (int)((uint32_t)(cl + 1) * (uint32_t)T / (uint32_t)ncl) : (int)((int64_t)(cl + 1) * T / ncl);
    const int ntile = t1 - t0;  // units of this CTA
    const int njb = NB / JB;
    const int jb0 = rank * njb / C, jb1 = (rank + 1) * njb / C;
    const int jpt = jb1 - jb0;  // jobs per unit
    const int J = ntile * jpt;
    const int j0 = warp * J / W, j1 = (warp + 1) * J / W;
    const int n_jobs = j1 - j0;
    const QmSmem sl = qm_smem(M, S, JB, TL, a.nkb_max, C > 1 ? a.out_tiles : 0);
    // (debug build: the layout must fit the launch's shared memory; every CTA
    // of a cluster decides alike)
    if (!QG_OK(sl.bytes <= dynamic_smem_bytes(), timeouts, 910)) return;
    float* outb = reinterpret_cast<float*>(smem + sl.out);
    int* tab = reinterpret_cast<int*>(smem + sl.tab);
    uint64_t* wbar = reinterpret_cast<uint64_t*>(smem + sl.bar) + warp * S;
    uint64_t* abar = reinterpret_cast<uint64_t*>(smem + sl.bar) + W * S;  // the activation copy
    const uint32_t wnib = sb + sl.nib + (uint32_t)(warp * S) * NIB;  // this warp's ring (shared addresses)
    const uint32_t wds = sb + sl.ds + (uint32_t)(warp * S) * DSB;
    uint8_t* wnib_p = smem + sl.nib + (size_t)warp * S * NIB;
    uint8_t* wds_p = smem + sl.ds + (size_t)warp * S * DSB;

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&wbar[s], 1);
        if (warp == 0) mbar_init(abar, 1);
        fence_barrier_init();
    }
    if (warp == 1 && lane < (PAIR ? 4 : 2)) {
        const CUtensorMap* map = lane == 0 ? &tn0 : lane == 1 ? &td0 : lane == 2 ? &tn1 : &td1;
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
    }

    // The copy cursor: job ikj of the unit whose first group is igrp (of the
    // second weight when isec), job ikg of the row (JB-block unit).
    int ikj, ikg, igrp;
    bool isec;
    int tl, kj;  // the job being worked on: unit (CTA-local) and job within it
    {
        const int tau = jpt > 0 ? j0 / jpt : 0;
        tl = tau;
        kj = j0 - tau * jpt;
        const int tg = t0 + tau;
        ikj = kj;
        ikg = jb0 + kj;
        isec = PAIR && tg >= U1;
        igrp = (isec ? tg - U1 : tg) * UG;
    }
    __syncthreads();  // barriers initialized
    const uint64_t pol = __shfl_sync(FULL, l2_evict_first_policy(), 0);

    int issued = 0, iss_slot = 0;
    // test only: the job whose copy is never issued, so that its wait runs out
    // (job 0 of CTA 0, in the warp that holds it)
    const int dropped = a.drop_copy && blockIdx.x == 0 && j0 == 0 && j1 > 0 ? 0 : -1;
    auto issue = [&]() {
        const int h = ikg & (JPC - 1), c = ikg >> JPC_LOG;  // which JB blocks of which 32-block chunk
        // (debug build: a job outside its weight completes its stage empty)
        const bool ok =
            QG_OK(igrp >= 0 && igrp < (isec ? a.N2 : a.N) / GROUP && c < (NB + CHUNK - 1) / CHUNK, timeouts, 901);
        if (lane == 0 && issued != dropped) {
            uint64_t* bar = &wbar[iss_slot];
            uint8_t* dst = wnib_p + (size_t)iss_slot * NIB;
            fence_proxy_async();
            mbar_arrive_expect_tx(bar, ok ? NIB + DSB : 0u);
            const CUtensorMap* map = isec ? &tn1 : &tn0;
            if (ok) {
                tma_load_4d(dst, map, h * JB * 16, 0, c, igrp, bar, pol);
                if (JB > TC_LINE_JB) tma_load_4d(dst + TC_BOX, map, h * JB * 16 + 128, 0, c, igrp, bar, pol);
                tma_load_3d(wds_p + (size_t)iss_slot * DSB, isec ? &td1 : &td0, h * JB * 8, c, igrp, bar, pol);
            }
        }
        ++ikg;
        if (++ikj == jpt) {  // next unit
            ikj = 0;
            ikg = jb0;
            igrp += UG;
            if (PAIR && !isec && igrp == U1 * UG) {
                isec = true;
                igrp = 0;
            }
        }
        ++issued;
        if (++iss_slot == S) iss_slot = 0;
    };
    pdl_wait();
    // The activation's K part first (every job needs it): one bulk copy per
    // row into the tail of the B-fragment region, read back before the
    // records overwrite it; then the ring's copies.
    const uint32_t act = sb + sl.act, meta = sb + sl.meta;
    const int nkb = jpt * JB;
    const uint32_t row_bytes = (uint32_t)nkb * Q8_1_BYTES, rstride = row_bytes + 16;
    const uint32_t raw_off = sl.act + (uint32_t)a.nkb_max * M * 64 - (uint32_t)M * rstride;
    if (threadIdx.x == 0 && row_bytes > 0) {
        const bool ok = QG_OK(qg_in(((int64_t)(M - 1) * NB + (int64_t)jb0 * JB) * Q8_1_BYTES, row_bytes,
                                    (int64_t)M * NB * Q8_1_BYTES),
                              timeouts, 902);
        mbar_arrive_expect_tx(abar, ok ? (uint32_t)M * row_bytes : 0u);
        for (int n = 0; ok && n < M; ++n)
            bulk_g2s_plain(smem + raw_off + (size_t)n * rstride,
                           a.xq + ((int64_t)n * NB + (int64_t)jb0 * JB) * Q8_1_BYTES, row_bytes, abar);
    }
    while (issued < n_jobs && issued < S) issue();

    if (warp == W - 1) {
        // Units cut by a warp boundary (found at the first boundary strictly
        // inside them): the unit, the warps holding its pieces (a mask), and
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
    bool alive = true;
    if (row_bytes > 0 && !__all_sync(FULL, mbar_wait_bounded(abar, 0))) {
        if (lane == 0) atomicAdd_system(timeouts, 1u);
        alive = false;
    }
    alive = __syncthreads_and(alive);
    if (alive) {
        uint32_t xw[QM_UNITS][9];
        qm_stage_load<M>(xw, sb + raw_off, (int)rstride, nkb);
        __syncthreads();  // the raw bytes are all read
        qm_stage_store<M>(xw, act, meta, nkb);
    }
    __syncthreads();  // the activation is staged

    // The lane's constant parts of the job addresses.
    const uint32_t L = (uint32_t)((lane & 7) + 8 * ((lane >> 3) & 1));
    const uint32_t cpiece = (uint32_t)(((lane >> 4) & 1) ^ (lane & 7));
    const uint32_t ld_off = L * 128u + (cpiece << 4);
    const uint32_t sc_off = (uint32_t)((g >> 2) * JB * 8 + (g & 3) * 2);
    const uint32_t bA0 = act + (uint32_t)((g < M ? g : M - 1) * 64 + t * 16);
    const uint32_t bM0 = meta + (uint32_t)(t * 16);

    float acc[TL][4];
    // A warp's pieces of cut units (its first segment, its last) wait in
    // registers until the loop ends; they go to the ring area afterwards.
    float first_piece[TL][4];
#pragma unroll
    for (int u = 0; u < TL; ++u)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[u][i] = first_piece[u][i] = 0.0f;
    bool has_first = false, has_last = false;
    int slot = 0, consumed = 0, seg_begin = j0;
    uint32_t phase = 0;
    for (int j = j0; alive && j < j1; ++j) {
        if (!__all_sync(FULL, mbar_wait_bounded(&wbar[slot], phase))) {
            if (lane == 0) atomicAdd_system(timeouts, 1u);
            alive = false;
            break;
        }
        ++consumed;
        qm_job<M, JB, TL>(wnib + (uint32_t)slot * NIB + ld_off, wds + (uint32_t)slot * DSB + sc_off,
                          bA0 + (uint32_t)kj * (JB * M * 64), bM0 + (uint32_t)kj * (JB * 96), acc);
        __syncwarp();
        if (issued < n_jobs) issue();  // into the stage just read
        if (++slot == S) {
            slot = 0;
            phase ^= 1u;
        }
        const bool unit_end = ++kj == jpt;
        if (unit_end || j + 1 == j1) {
            // a segment of unit tl ends: whole units go out; a piece of a cut
            // unit is the warp's first segment (kept) or its last (left in acc)
            const bool whole = unit_end && seg_begin == tl * jpt;
            if (whole || seg_begin == j0) {
#pragma unroll
                for (int u = 0; u < TL; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int v = u * QM_VT + lane * 4 + i;
                        if (!whole) first_piece[u][i] = acc[u][i];
                        else if (C > 1) outb[(size_t)tl * VU + v] = acc[u][i];
                        else qm_store<M, TL>(a, U1, t0 + tl, v, acc[u][i]);
                        acc[u][i] = 0.0f;
                    }
                has_first = has_first || !whole;
            } else {
                has_last = true;  // ends at j1: the loop ends with it
            }
            seg_begin = j + 1;
            if (unit_end) {
                ++tl;
                kj = 0;
            }
        }
    }
    // After a timeout, give the copies still in flight a bounded wait before
    // the shared memory is released.
    if (lane == 0) {
        for (int jj = consumed; jj < issued; ++jj)
            if (jj != dropped) mbar_wait_bounded(&wbar[jj % S], (uint32_t)((jj / S) & 1));
        if (!alive && warp == 0) mbar_wait_bounded(abar, 0);
    }
    alive = __syncthreads_and(alive);  // the ring area is free
    float* slots = reinterpret_cast<float*>(smem + sl.nib);  // [warp][first, last][VU floats]
#pragma unroll
    for (int u = 0; u < TL; ++u)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int v = u * QM_VT + lane * 4 + i;
            if (has_first) slots[(size_t)(warp * 2) * VU + v] = first_piece[u][i];
            if (has_last) slots[(size_t)(warp * 2 + 1) * VU + v] = acc[u][i];
        }
    __syncthreads();

    // Units cut by a warp boundary: their pieces added in warp order.
    const int ne = alive ? tab[0] : 0;
    for (int o = threadIdx.x; o < ne * VU; o += QM_THREADS) {
        const int e = o / VU, v = o - e * VU;
        const int tau = tab[1 + 3 * e];
        unsigned mask = (unsigned)tab[2 + 3 * e];
        const int wa = __ffs(mask) - 1;
        float sum = slots[(size_t)(wa * 2 + tab[3 + 3 * e]) * VU + v];
        mask &= mask - 1;
        while (mask) {
            const int ww = __ffs(mask) - 1;
            mask &= mask - 1;
            sum += slots[(size_t)(ww * 2) * VU + v];
        }
        if (C > 1) outb[(size_t)tau * VU + v] = sum;
        else qm_store<M, TL>(a, U1, t0 + tau, v, sum);
    }
    if (C > 1) {
        // The K parts of each unit, added in rank order; rank r writes its
        // share of the cluster's units.
        cluster_sync_all();
        const int ta = rank * ntile / C, tb = (rank + 1) * ntile / C;
        for (int o = threadIdx.x; alive && o < (tb - ta) * VU; o += QM_THREADS) {
            const int tau = ta + o / VU, v = o - (tau - ta) * VU;
            const float* p = outb + (size_t)tau * VU + v;
            float sum = ld_dsmem_f32(p, 0);
            for (int rr = 1; rr < C; ++rr) sum += ld_dsmem_f32(p, (uint32_t)rr);
            qm_store<M, TL>(a, U1, t0 + tau, v, sum);
        }
        cluster_sync_all();  // no CTA leaves while its shared memory is read
    }
}

}  // namespace qgemv
