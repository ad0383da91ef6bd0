// Shared device-side definitions of the GB300 small-M block-quantized GEMV
// library: packed weight layouts, the Q8_1 block, the shared-memory
// activation tile, integer block dots and the top-1 key.
//
// The pages ("Qwen3.6 27B Q4_0 DFlash/SYCL closure", "Q6_K M=6 fused DFlash
// top-1 production record", "Qwen3.6 27B B70 follow-up: Q8 activation cache")
// name Q4_0, Q6_K and Q8_1 but do not define their bytes; the definitions used
// are the llama.cpp-family ones:
//   Q8_1  per 32 activations: fp16 d, fp16 s = d * sum(q), int8 q[32]   (36 B)
//   Q4_0  per 32 weights:     fp16 d, 4-bit q, value d * (q - 8)         (18 B)
//   Q6_K  per 256 weights:    fp16 d, int8 sc[16], 6-bit q,
//                             value d * sc[i / 16] * (q - 32)           (210 B)
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qgemv {

constexpr int QK = 32;              // values per Q8_1 / Q4_0 block
constexpr int QK_K = 256;           // values per Q6_K superblock
constexpr int Q8_1_BYTES = 36;
constexpr int Q4_0_BYTES = 18;
constexpr int Q6_K_BYTES = 210;
constexpr int MAX_M = 17;

// ---------------------------------------------------------------------------
// Debug build (compiled with -DQGEMV_BOUNDS_CHECK): explicit checks of the
// indexes the kernels compute for their global and shared-memory accesses,
// against the extents their arguments imply.  A failing check skips the
// access (a skipped copy still completes its mbarrier stage, with no bytes)
// and records itself in the library's status page: word 1 counts failures,
// word 2 keeps the site number of the first.  `status` is that page (word 0
// is the wait-timeout count).  No assert, no trap: the kernel runs on.  In
// the release build QG_OK is the constant true and every check compiles away.
// ---------------------------------------------------------------------------
#ifdef QGEMV_BOUNDS_CHECK
static __device__ __noinline__ void qg_bounds_fail(unsigned int* status, unsigned int site)
{
    if (atomicAdd_system(status + 1, 1u) == 0u) atomicExch_system(status + 2, site);
}
__device__ __forceinline__ bool qg_ok(bool ok, unsigned int* status, unsigned int site)
{
    if (!ok && status) qg_bounds_fail(status, site);
    return ok;
}
#define QG_OK(cond, status, site) ::qgemv::qg_ok((cond), (status), (site))
#else
#define QG_OK(cond, status, site) true
#endif

// [lo, lo + n) lies within [0, extent) (64-bit byte or element offsets).
__host__ __device__ __forceinline__ bool qg_in(int64_t lo, int64_t n, int64_t extent)
{
    return lo >= 0 && n >= 0 && lo + n <= extent;
}

// ---------------------------------------------------------------------------
// Packed weight layouts.  Rows are taken in groups of 4 (the last group may
// hold fewer) and each row of NB = K/32 blocks is cut into chunks of 32
// blocks (the last chunk may be shorter, nb_tail blocks).  One (group, chunk)
// is one contiguous, 16-byte-aligned region, so the chunk of a row group is
// fetched with a single bulk copy, and a whole group is contiguous too.
// Groups follow one another; inside a group the chunks follow one another.
//
// Q4_0 group-chunk of `rows` rows and nb blocks:
//   nib[rows][nb] (16 B each: the canonical qs bytes of the block, unchanged)
//   d[nb][rows] (fp16 bits, copied raw), zero padded to 16 B.
//   4 rows x 32 blocks = 2048 + 256 = 2304 B.  Row-major codes let the 32
//   lanes of a warp (one block each) read 512 consecutive bytes per row; the
//   block-major scales put the four rows of one block next to each other, so
//   a lane reads its block's four scales with one 8-byte load.
// Q6_K group-chunk (nb a multiple of 8), row-major: per row one tile
//   ql[nb] 16 B: byte t = low4(q[t]) | low4(q[t + 16]) << 4
//   qh[nb]  8 B: byte t, bits 2s..2s+1 = high2(q[t + 8 s]), s = 0..3
//   sc[nb]  2 B: the int8 subscales of the block's two 16-value halves
// then the fp16 superblock scales of the chunk, d[rows][nb / 8], zero padded
// to 16 B;  full row tile 832 B, group-chunk 4 * 832 + 32 = 3360 B.
// For N % 4 == 0 and K % 1024 == 0 there is no padding and the pack has
// exactly the canonical size (18 B per Q4_0 block, 210 B per Q6_K superblock).
// ---------------------------------------------------------------------------

constexpr int CHUNK = 32;  // blocks per chunk
constexpr int GROUP = 4;   // rows per group

__host__ __device__ inline int pad16(int v) { return (v + 15) & ~15; }

struct Layout {
    int fmt;            // 0 = Q4_0, 1 = Q6_K
    int N, NB, nch, nb_tail;
    int64_t n_groups;
    __host__ __device__ int nb(int c) const { return c == nch - 1 ? nb_tail : CHUNK; }
    // Q6_K: bytes of one row's tile in chunk c
    __host__ __device__ int tile(int c) const { return nb(c) * 26; }
    __host__ __device__ int chunk_bytes(int rows, int c) const
    {
        const int n = nb(c);
        return fmt == 0 ? rows * n * 16 + pad16(rows * n * 2) : rows * n * 26 + pad16(rows * (n / 8) * 2);
    }
    __host__ __device__ int64_t group_bytes(int rows) const
    {
        return (int64_t)(nch - 1) * chunk_bytes(rows, 0) + chunk_bytes(rows, nch - 1);
    }
    __host__ __device__ int rows_in(int64_t g) const
    {
        const int64_t r = (int64_t)N - g * GROUP;
        return r < GROUP ? (int)r : GROUP;
    }
    // every group but the last is full
    __host__ __device__ int64_t group_offset(int64_t g) const { return g * group_bytes(GROUP); }
    __host__ __device__ int64_t chunk_offset(int64_t g, int c) const
    {
        return group_offset(g) + (int64_t)c * chunk_bytes(rows_in(g), 0);
    }
    __host__ __device__ int64_t total_bytes() const
    {
        return group_offset(n_groups - 1) + group_bytes(rows_in(n_groups - 1));
    }
};

__host__ __device__ inline Layout make_layout(int fmt, int N, int K)
{
    Layout L;
    L.fmt = fmt;
    L.N = N;
    L.NB = K / QK;
    L.nch = (L.NB + CHUNK - 1) / CHUNK;
    L.nb_tail = L.NB - (L.nch - 1) * CHUNK;
    L.n_groups = ((int64_t)N + GROUP - 1) / GROUP;
    return L;
}

// Where the pieces of block b of row n live.
struct BlockAddr {
    const uint8_t* q;   // Q4_0: the 16 code bytes;  Q6_K: the code bytes P (16 B)
    const uint8_t* qh;  // Q6_K: the code bytes Q (8 B)
    const uint8_t* sc;  // Q6_K: the two subscales
    const uint8_t* d;   // fp16 scale (Q4_0: the block's; Q6_K: the superblock's)
};

__host__ __device__ inline BlockAddr block_addr(const void* base, const Layout& L, int64_t n, int b)
{
    const int64_t g = n / GROUP;
    const int c = b / CHUNK;
    const int rows = L.rows_in(g);
    const int r = (int)(n - g * GROUP), j = b - c * CHUNK, nb = L.nb(c);
    const uint8_t* gc = static_cast<const uint8_t*>(base) + L.chunk_offset(g, c);
    BlockAddr a;
    if (L.fmt == 0) {
        a.q = gc + (r * nb + j) * 16;
        a.d = gc + nb * rows * 16 + (j * rows + r) * 2;
        a.qh = a.sc = nullptr;
    } else {
        const uint8_t* t = gc + r * nb * 26;
        a.q = t + j * 16;
        a.qh = t + nb * 16 + j * 8;
        a.sc = t + nb * 24 + j * 2;
        a.d = gc + rows * nb * 26 + (r * (nb / 8) + j / 8) * 2;
    }
    return a;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch (the library's kernels are launched with
// programmatic stream serialization): a kernel lets the next kernel of the
// stream be scheduled as soon as it starts, and waits for the previous one
// (its completion and memory) before touching anything that kernel may
// write or read.  Only L2 prefetches of weights run before the wait: they
// cannot observe stale data, since writes are made in L2.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Loads
// ---------------------------------------------------------------------------

// Streaming read-only 16-byte load: weights are read exactly once, so keep
// them out of L1.
__device__ __forceinline__ uint4 ld_stream_v4(const uint4* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint2 ld_stream_v2(const uint2* p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const void* p)
{
    uint16_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void prefetch_l2(const void* p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---------------------------------------------------------------------------
// Q8_1 quantization of one 32-value block by one thread.
// d = max|x| / 127 (IEEE fp32 divide), q_i = round(x_i / d) with round half
// away from zero; an all-zero block gives d = 0 and q = 0.  The stored scale is
// the fp16 rounding (nearest even) of d; x is divided by the fp32 d.
// ---------------------------------------------------------------------------

struct Q81Block {
    uint32_t q[8];  // codes, 4 per word, value order
    float d;        // fp32 scale (before fp16 rounding)
    int s_lo, s_hi; // sum of codes 0..15 and 16..31
};

// xb: 32 consecutive fp32 values; vec4: xb is 16-byte aligned.
__device__ __forceinline__ void q8_1_quantize_block(const float* xb, bool vec4, Q81Block& o)
{
    float v[32];
    if (vec4) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 f = reinterpret_cast<const float4*>(xb)[k];
            v[4 * k + 0] = f.x;
            v[4 * k + 1] = f.y;
            v[4 * k + 2] = f.z;
            v[4 * k + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = xb[k];
    }
    float amax = 0.0f;
#pragma unroll
    for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(v[k]));
    o.d = __fdiv_rn(amax, 127.0f);
    int s0 = 0, s1 = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        uint32_t word = 0;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            int q = 0;
            if (amax != 0.0f) {
                q = (int)roundf(__fdiv_rn(v[4 * w + t], o.d));
                q = max(-127, min(127, q));
            }
            word |= ((uint32_t)q & 0xFFu) << (8 * t);
            if (w < 4) s0 += q; else s1 += q;
        }
        o.q[w] = word;
    }
    o.s_lo = s0;
    o.s_hi = s1;
}

// The same quantization of one 32-value block by 8 consecutive lanes of a
// warp (lanes 8k .. 8k+7; sub = lane & 7 holds values 4 sub .. 4 sub + 3).
// Every lane of the warp must call it (full-warp shuffles).  The maximum, the
// divides and the rounding are the single-thread routine's, so the codes and
// scales are bit-identical to it.
struct Q81Lanes {
    uint32_t word;  // codes 4 sub .. 4 sub + 3 (word `sub` of the block's codes)
    float d;        // fp32 scale (before fp16 rounding), same in all 8 lanes
    int s_half;     // sum of codes 0..15 (sub < 4) or 16..31 (sub >= 4)
    int s_all;      // sum of all 32 codes
};

__device__ __forceinline__ Q81Lanes q8_1_quantize_8lanes(const float4 v)
{
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    Q81Lanes o;
    o.d = __fdiv_rn(amax, 127.0f);
    int q0 = 0, q1 = 0, q2 = 0, q3 = 0;
    if (amax != 0.0f) {
        q0 = max(-127, min(127, (int)roundf(__fdiv_rn(v.x, o.d))));
        q1 = max(-127, min(127, (int)roundf(__fdiv_rn(v.y, o.d))));
        q2 = max(-127, min(127, (int)roundf(__fdiv_rn(v.z, o.d))));
        q3 = max(-127, min(127, (int)roundf(__fdiv_rn(v.w, o.d))));
    }
    o.word = ((uint32_t)q0 & 0xFFu) | (((uint32_t)q1 & 0xFFu) << 8) | (((uint32_t)q2 & 0xFFu) << 16) |
             ((uint32_t)q3 << 24);
    int s = q0 + q1 + q2 + q3;
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    o.s_half = s;
    o.s_all = s + __shfl_xor_sync(0xffffffffu, s, 4);
    return o;
}

// Four values of a block for q8_1_quantize_8lanes (vec4: p is 16-byte aligned).
__device__ __forceinline__ float4 load_4_values(const float* p, bool vec4)
{
    if (vec4) return *reinterpret_cast<const float4*>(p);
    return make_float4(p[0], p[1], p[2], p[3]);
}

// ---------------------------------------------------------------------------
// Shared-memory activation tile (one CTA, a chunk of KC blocks, M rows).
//   aq  [M][2][KC] uint4 : q bytes 0..15 (h = 0) and 16..31 (h = 1) of block b
//   am  [M][KC]    uint2 : x = fp32 bits of the block's fp16 scale d_a
//                          y = Q4_0: -8 * sum(q[0..31])
//                              Q6_K: sum(q[0..15]) | sum(q[16..31]) << 16 (int16 pair)
// The integer sums fold the weight offsets (q_w - 8, q_w - 32) into the dot
// products exactly: sum (q_w - c) q_a = sum q_w q_a - c * sum q_a.
// Lanes of a warp read consecutive blocks, so the 16-byte reads are
// bank-conflict free.
// ---------------------------------------------------------------------------

constexpr int ACT_BYTES_PER_BLOCK = 2 * 16 + 8;  // per (row, block)

enum WeightFormat { FMT_Q4_0 = 0, FMT_Q6_K = 1 };

template <int FMT>
__device__ __forceinline__ uint32_t act_meta_sums(const uint32_t (&q)[8])
{
    int s0 = 0, s1 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) s0 = __dp4a((int)q[i], 0x01010101, s0);
#pragma unroll
    for (int i = 4; i < 8; ++i) s1 = __dp4a((int)q[i], 0x01010101, s1);
    if (FMT == FMT_Q4_0) return (uint32_t)(-8 * (s0 + s1));
    return ((uint32_t)s0 & 0xFFFFu) | ((uint32_t)s1 << 16);
}

template <int FMT>
__device__ __forceinline__ uint32_t act_meta_from_sums(int s_lo, int s_hi)
{
    if (FMT == FMT_Q4_0) return (uint32_t)(-8 * (s_lo + s_hi));
    return ((uint32_t)s_lo & 0xFFFFu) | ((uint32_t)s_hi << 16);
}

// Read one canonical Q8_1 block from global memory (4-byte aligned) into the
// tile representation.
template <int FMT>
__device__ __forceinline__ void act_from_q8_1(const uint8_t* blk, uint4& lo, uint4& hi, uint2& meta)
{
    const uint32_t* w = reinterpret_cast<const uint32_t*>(blk);
    uint32_t q[8];
    uint32_t ds = w[0];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = w[1 + i];
    lo = make_uint4(q[0], q[1], q[2], q[3]);
    hi = make_uint4(q[4], q[5], q[6], q[7]);
    float d = __half2float(__ushort_as_half((unsigned short)(ds & 0xFFFFu)));
    meta.x = __float_as_uint(d);
    meta.y = act_meta_sums<FMT>(q);
}

// ---------------------------------------------------------------------------
// Integer block dots.  All sums are exact in int32.
// ---------------------------------------------------------------------------

// Q4_0: the 8 words of codes (value order matching the activation words):
// word i < 4 = low nibbles of nib word i, word i + 4 = high nibbles.
__device__ __forceinline__ void q4_0_unpack(const uint4 nib, uint32_t (&w)[8])
{
    const uint32_t m = 0x0F0F0F0Fu;
    w[0] = nib.x & m;
    w[1] = nib.y & m;
    w[2] = nib.z & m;
    w[3] = nib.w & m;
    w[4] = (nib.x >> 4) & m;
    w[5] = (nib.y >> 4) & m;
    w[6] = (nib.z >> 4) & m;
    w[7] = (nib.w >> 4) & m;
}

// I = sum_i (q_w - 8) * q_a, starting from init = -8 * sum(q_a) + bias.
__device__ __forceinline__ int q4_0_dot(const uint32_t (&w)[8], const uint4 lo, const uint4 hi, int init)
{
    int s = init;
    s = __dp4a((int)w[0], (int)lo.x, s);
    s = __dp4a((int)w[1], (int)lo.y, s);
    s = __dp4a((int)w[2], (int)lo.z, s);
    s = __dp4a((int)w[3], (int)lo.w, s);
    s = __dp4a((int)w[4], (int)hi.x, s);
    s = __dp4a((int)w[5], (int)hi.y, s);
    s = __dp4a((int)w[6], (int)hi.z, s);
    s = __dp4a((int)w[7], (int)hi.w, s);
    return s;
}

// Q6_K: the 8 words of one packed 32-value block (the pack's per-row,
// per-block 24 code bytes: P[16], byte t = q_t | high2(q_{16+t}) << 6, and
// Q[8], byte u = low4(q_{16+u}) | low4(q_{24+u}) << 4).  Words 0..3 hold the
// codes q_0 .. q_15 (values 4i .. 4i+3 in word i); words 4..7 hold 4 q_16 ..
// 4 q_31, each code times four, which puts its low four bits next to its high
// two without a shift of P.  The factor four is taken out of the second
// half's dot product by the caller (q6_k_dot_init).
__device__ __forceinline__ void q6_k_unpack(const uint4 P, const uint2 Q, uint32_t (&w)[8])
{
    const uint32_t m6 = 0x3F3F3F3Fu, mh = 0xC0C0C0C0u, ml = 0x3C3C3C3Cu;
    w[0] = P.x & m6;
    w[1] = P.y & m6;
    w[2] = P.z & m6;
    w[3] = P.w & m6;
    w[4] = (P.x & mh) | ((Q.x << 2) & ml);
    w[5] = (P.y & mh) | ((Q.y << 2) & ml);
    w[6] = (P.z & mh) | ((Q.x >> 2) & ml);
    w[7] = (P.w & mh) | ((Q.y >> 2) & ml);
}

// d = dot of the four unsigned bytes of a with the four signed bytes of b, plus c.
__device__ __forceinline__ int dp4a_u8s8(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The two 16-value half-block dp4a chains of a Q6_K block, continued from
// the starts g0 and g1: g0 += sum_{i<16} q_i q_a[i], g1 += sum_{i>=16} 4 q_i q_a[i].
__device__ __forceinline__ void q6_k_half_dots(const uint32_t (&w)[8], const uint4 lo, const uint4 hi, int& g0, int& g1)
{
    g0 = __dp4a((int)w[0], (int)lo.x, g0);
    g0 = __dp4a((int)w[1], (int)lo.y, g0);
    g0 = __dp4a((int)w[2], (int)lo.z, g0);
    g0 = __dp4a((int)w[3], (int)lo.w, g0);
    g1 = dp4a_u8s8(w[4], hi.x, g1);
    g1 = dp4a_u8s8(w[5], hi.y, g1);
    g1 = dp4a_u8s8(w[6], hi.z, g1);
    g1 = dp4a_u8s8(w[7], hi.w, g1);
}

// 4 J, J = sc0 * sum_{i<16} (q_i - 32) q_a[i] + sc1 * sum_{i>=16} (q_i - 32) q_a[i]
// exactly (|4 J| < 2^27), with the offsets folded into the chain starts:
// g0 = -32 * sum(q_a[0..15]), g1 = -128 * sum(q_a[16..31]) (the second half's
// codes come four times over); sc0x4 = 4 * sc0, sc1 = the block's two int8
// subscales.
__device__ __forceinline__ int q6_k_dot_init(const uint32_t (&w)[8], const uint4 lo, const uint4 hi, int g0, int g1,
                                             int sc0x4, int sc1)
{
    q6_k_half_dots(w, lo, hi, g0, g1);
    return sc0x4 * g0 + sc1 * g1;
}

// The same 4 J, from the packed activation sums (sum(q_a[0..15]) |
// sum(q_a[16..31]) << 16, int16 pair) and the two subscale bytes sc2.
__device__ __forceinline__ int q6_k_dot(const uint32_t (&w)[8], const uint4 lo, const uint4 hi, uint32_t sums,
                                        uint32_t sc2)
{
    return q6_k_dot_init(w, lo, hi, -32 * (int)(int16_t)(sums & 0xFFFFu), -128 * (int)(int16_t)(sums >> 16),
                         4 * (int)(int8_t)(sc2 & 0xFFu), (int)(int8_t)((sc2 >> 8) & 0xFFu));
}

// Packed fp32 pairs (sm_100 and later): (ax, ay) = (bx, by) * (cx, cy) + (ax, ay),
// (dx, dy) = (bx, by) * (cx, cy) and (dx, dy) = (bx, by) + (cx, cy), each
// lane one IEEE fma / mul / add, so the results equal the scalar ones bit for
// bit with half the instructions.
__device__ __forceinline__ void fma_f32x2(float& ax, float& ay, float bx, float by, float cx, float cy)
{
    asm("{\n\t.reg .b64 a, b, c;\n\t"
        "mov.b64 a, {%0, %1};\n\tmov.b64 b, {%2, %3};\n\tmov.b64 c, {%4, %5};\n\t"
        "fma.rn.f32x2 a, b, c, a;\n\tmov.b64 {%0, %1}, a;\n\t}"
        : "+f"(ax), "+f"(ay)
        : "f"(bx), "f"(by), "f"(cx), "f"(cy));
}

__device__ __forceinline__ void mul_f32x2(float& dx, float& dy, float bx, float by, float cx, float cy)
{
    asm("{\n\t.reg .b64 d, b, c;\n\t"
        "mov.b64 b, {%2, %3};\n\tmov.b64 c, {%4, %5};\n\t"
        "mul.rn.f32x2 d, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(dx), "=f"(dy)
        : "f"(bx), "f"(by), "f"(cx), "f"(cy));
}

__device__ __forceinline__ void add_f32x2(float& dx, float& dy, float bx, float by, float cx, float cy)
{
    asm("{\n\t.reg .b64 d, b, c;\n\t"
        "mov.b64 b, {%2, %3};\n\tmov.b64 c, {%4, %5};\n\t"
        "add.rn.f32x2 d, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(dx), "=f"(dy)
        : "f"(bx), "f"(by), "f"(cx), "f"(cy));
}

// Exact int -> float for |i| < 2^22 without a conversion instruction: the
// integer is added to the bit pattern of 1.5 * 2^23, whose unit in the last
// place is 1.  Used by the Q4_0 path, where |I| <= 32 * 8 * 127.
constexpr int MAGIC_I2F_BITS = 0x4B400000;
constexpr float MAGIC_I2F = 12582912.0f;

// ---------------------------------------------------------------------------
// Top-1 key: orders (value, index) pairs so that a 64-bit max picks the
// largest value and, among exactly equal values, the lowest index.  -0 and +0
// are the same value; NaN maps to 0 and so never wins; when every value of a
// row is NaN the result is index 0.  ("Q6_K M=6 fused DFlash top-1 production
// record", Exactness and safety contracts, item 3: lowest-token-ID
// finite-tie contract shared by the fused reducer and the generic argmax.)
// ---------------------------------------------------------------------------

__device__ __forceinline__ unsigned long long top1_key(float v, int n)
{
    if (v != v) return 0ull;
    uint32_t u = (v == 0.0f) ? 0u : __float_as_uint(v);
    uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)n);
}

__host__ __device__ inline int top1_key_to_id(unsigned long long k)
{
    return k == 0ull ? 0 : (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
}

// The fp32 value a top-1 key was made from (+0 for a zero; NaN for key 0,
// i.e. a row that held only NaN).
__device__ __forceinline__ float top1_key_to_value(unsigned long long k)
{
    if (k == 0ull) return __int_as_float(0x7fffffff);
    const uint32_t ord = (uint32_t)(k >> 32);
    return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        unsigned long long t = __shfl_xor_sync(0xffffffffu, v, o);
        v = t > v ? t : v;
    }
    return v;
}

// Cross-CTA top-1 workspace: M 64-bit keys, then a CTA completion counter.
// Every call leaves it zeroed again (the last CTA resets it).
struct Top1Workspace {
    unsigned long long keys[MAX_M];
    unsigned int done;
    unsigned int pad;
};

}  // namespace qgemv
