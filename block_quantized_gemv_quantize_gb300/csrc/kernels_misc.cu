// Q8_1 activation quantizer, weight repackers, row argmax (the unfused
// control path) and the integer block-dot debug kernel.
#include "launch.cuh"

namespace qgemv {

DeviceInfo device_info()
{
    static DeviceInfo cache[64];
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DeviceInfo{0, 0};
    std::call_once(once[dev], [&]() {
        DeviceInfo d{0, 0};
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            d = DeviceInfo{0, 0};
        cache[dev] = d;
    });
    return cache[dev];
}

// ---------------------------------------------------------------------------
// quantize_q8_1: eight lanes per 32-value block, four blocks per warp step
// ("Qwen3.6 27B B70 follow-up: Q8 activation cache", Q8_1 activation cache
// prototype: the activation is quantized once and the Q8_1 copy is reused by
// sibling matmuls).  Lane sub of a block writes code word sub; lane 0 of the
// block also writes the fp16 pair (d, s).
// ---------------------------------------------------------------------------

constexpr int QUANT_THREADS = 128;

__global__ void __launch_bounds__(QUANT_THREADS) quantize_q8_1_kernel(const float* __restrict__ x, int64_t ldx,
                                                                      uint8_t* __restrict__ xq, int M, int NB,
                                                                      unsigned int* st)
{
    pdl_launch_dependents();
    pdl_wait();
    const int64_t nblk = (int64_t)M * NB;
    const bool vec4 = ((reinterpret_cast<uintptr_t>(x) | ((uintptr_t)ldx * 4)) & 15u) == 0;
    const int lane = threadIdx.x & 31, sub = lane & 7;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t i0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 4; i0 < nblk;
         i0 += warps * 4) {  // warp-uniform
        const int64_t mine = i0 + (lane >> 3);
        const int64_t i = mine < nblk ? mine : nblk - 1;  // spare lanes redo the last block, unwritten
        const int m = (int)(i / NB), b = (int)(i - (int64_t)m * NB);
        const int64_t xo = (int64_t)m * ldx + (int64_t)b * QK + 4 * sub;
        float4 xv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (QG_OK(qg_in(xo, 4, (int64_t)(M - 1) * ldx + (int64_t)NB * QK), st, 101)) xv = load_4_values(x + xo, vec4);
        const Q81Lanes o = q8_1_quantize_8lanes(xv);
        if (mine < nblk && QG_OK(qg_in(mine * Q8_1_BYTES, Q8_1_BYTES, nblk * Q8_1_BYTES), st, 102)) {
            uint32_t* blk = reinterpret_cast<uint32_t*>(xq + mine * Q8_1_BYTES);  // 4-byte aligned
            blk[1 + sub] = o.word;
            if (sub == 0) {
                const __half d16 = __float2half_rn(o.d);
                const __half s16 = __float2half_rn(__fmul_rn(o.d, (float)o.s_all));
                blk[0] = (uint32_t)__half_as_ushort(d16) | ((uint32_t)__half_as_ushort(s16) << 16);
            }
        }
    }
}

int launch_quantize_q8_1(const float* x, int64_t ldx, void* xq, int M, int K, cudaStream_t s)
{
    const DeviceInfo di = device_info();
    if (di.sms <= 0) return QGEMV_CUDA_ERROR;
    const int NB = K / QK;
    const int64_t nblk = (int64_t)M * NB;
    const int64_t per_cta = (QUANT_THREADS / 32) * 4;  // blocks per CTA step
    int64_t grid = (nblk + per_cta - 1) / per_cta;
    if (grid > (int64_t)di.sms * 16) grid = (int64_t)di.sms * 16;
    if (launch_pdl(quantize_q8_1_kernel, dim3((unsigned)grid), dim3(QUANT_THREADS), 0, s, x, ldx,
                   static_cast<uint8_t*>(xq), M, NB, wait_timeout_counter()) != cudaSuccess)
        return QGEMV_CUDA_ERROR;
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

// ---------------------------------------------------------------------------
// RMSNorm fused with the Q8_1 quantizer ("Qwen3.6 27B Q4_0 DFlash/SYCL
// closure", Closed or negative paths: the down-to-next-RMSNorm/Q8
// boundary): one CTA of RMS_THREADS threads per row,
//   S = sum_k x_k^2 in fp32: thread t adds x_k * x_k for k = t, t + 512, ...
//       in increasing k (separate multiply and add, no contraction), then the
//       512 partial sums are added pairwise, t += t + h for h = 256, ..., 1;
//   r = 1 / sqrt(S / K + eps), x^_k = (x_k * r) * gamma_k, all fp32 IEEE;
// and x^ is quantized to Q8_1 exactly as quantize_q8_1 does.
// ---------------------------------------------------------------------------

constexpr int RMS_THREADS = 512;

__global__ void __launch_bounds__(RMS_THREADS) rmsnorm_quantize_q8_1_kernel(const float* __restrict__ x, int64_t ldx,
                                                                          const float* __restrict__ gamma, float eps,
                                                                          uint8_t* __restrict__ xq, int K,
                                                                          unsigned int* st)
{
    pdl_launch_dependents();
    pdl_wait();
    __shared__ float part[RMS_THREADS];
    __shared__ float s_r;
    const int m = blockIdx.x, t = threadIdx.x;
    const float* xr = x + (int64_t)m * ldx;
    float s = 0.0f;
    for (int k = t; k < K; k += RMS_THREADS)
        if (QG_OK(qg_in((int64_t)m * ldx + k, 1, (int64_t)(gridDim.x - 1) * ldx + K), st, 201))
            s = __fadd_rn(s, __fmul_rn(xr[k], xr[k]));
    part[t] = s;
    for (int h = RMS_THREADS / 2; h > 0; h >>= 1) {
        __syncthreads();
        if (t < h) part[t] = __fadd_rn(part[t], part[t + h]);
    }
    if (t == 0) s_r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(part[0], (float)K), eps)));
    __syncthreads();
    const float r = s_r;
    const int NB = K / QK, lane = t & 31, sub = lane & 7;
    const bool vec4 = ((reinterpret_cast<uintptr_t>(xr) | reinterpret_cast<uintptr_t>(gamma)) & 15u) == 0;
    for (int b0 = (t >> 5) * 4; b0 < NB; b0 += (RMS_THREADS / 32) * 4) {  // warp-uniform: 4 blocks per warp step
        const int mine = b0 + (lane >> 3);
        const int b = mine < NB ? mine : NB - 1;  // spare lanes redo the last block, unwritten
        float4 xv = make_float4(0.0f, 0.0f, 0.0f, 0.0f), gv = xv;
        if (QG_OK(qg_in((int64_t)b * QK + 4 * sub, 4, K), st, 202)) {
            xv = load_4_values(xr + (int64_t)b * QK + 4 * sub, vec4);
            gv = load_4_values(gamma + (int64_t)b * QK + 4 * sub, vec4);
        }
        const float4 v = make_float4(__fmul_rn(__fmul_rn(xv.x, r), gv.x), __fmul_rn(__fmul_rn(xv.y, r), gv.y),
                                     __fmul_rn(__fmul_rn(xv.z, r), gv.z), __fmul_rn(__fmul_rn(xv.w, r), gv.w));
        const Q81Lanes o = q8_1_quantize_8lanes(v);
        if (mine < NB &&
            QG_OK(qg_in(((int64_t)m * NB + mine) * Q8_1_BYTES, Q8_1_BYTES, (int64_t)gridDim.x * NB * Q8_1_BYTES), st,
                  203)) {
            uint32_t* blk = reinterpret_cast<uint32_t*>(xq + ((int64_t)m * NB + mine) * Q8_1_BYTES);
            blk[1 + sub] = o.word;
            if (sub == 0) {
                const __half d16 = __float2half_rn(o.d);
                const __half s16 = __float2half_rn(__fmul_rn(o.d, (float)o.s_all));
                blk[0] = (uint32_t)__half_as_ushort(d16) | ((uint32_t)__half_as_ushort(s16) << 16);
            }
        }
    }
}

int launch_rmsnorm_quantize_q8_1(const float* x, int64_t ldx, const float* gamma, float eps, void* xq, int M, int K,
                                 cudaStream_t s)
{
    if (launch_pdl(rmsnorm_quantize_q8_1_kernel, dim3(M), dim3(RMS_THREADS), 0, s, x, ldx, gamma, eps,
                   static_cast<uint8_t*>(xq), K, wait_timeout_counter()) != cudaSuccess)
        return QGEMV_CUDA_ERROR;
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

// ---------------------------------------------------------------------------
// Repackers: canonical blocks -> coalesced streams.  Pure bit moves; fp16
// scales are copied as raw bits ("Qwen3.6 27B Q4_0 DFlash/SYCL closure",
// Transfer, rule 7: converting fp16 storage objects numerically once produced
// an all-zero kernel).
// ---------------------------------------------------------------------------

// Q8_0 pack for the tensor-core kernel: per 16-row tile and job of 8 blocks
// one 4352-byte region = codes [block p][lane l = 4g + t][16 B] then scales
// [block p][row r] (fp16 bits).  Lane l's 16 bytes are values 2t, 2t+1,
// 2t+8, 2t+9, 16+2t, 17+2t, 24+2t, 25+2t of row g, then of row g + 8, each
// stored as q + 128 (q ^ 0x80).  Rows past N are zero codes and zero scales.
// One thread per (tile, block, lane); scales are raw bit copies.
__global__ void qpack_q8_0_kernel(const uint8_t* __restrict__ canon, uint8_t* __restrict__ pack, int N, int K,
                                  unsigned int* st)
{
    const int NB = K / QK, NJ = NB / 8;
    const int64_t T = (N + 15) / 16;
    const int64_t canon_bytes = (int64_t)N * NB * 34, pack_bytes = T * NJ * 4352;
    const int64_t total = T * NB * 32;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int l = (int)(i & 31);
        const int64_t tb = i >> 5;
        const int64_t tau = tb / NB;
        const int b = (int)(tb - tau * NB), j = b / 8, p = b % 8;
        const int g = l >> 2, t = l & 3;
        uint8_t* region = pack + (tau * NJ + j) * 4352;
        uint32_t words[4];
        for (int h = 0; h < 2; ++h) {
            const int64_t n = tau * 16 + g + 8 * h;
            const bool in = n < N && QG_OK(qg_in((n * NB + b) * 34, 34, canon_bytes), st, 301);
            const uint8_t* q = canon + (n * NB + b) * 34 + 2;
            const int e[8] = {2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9, 16 + 2 * t, 17 + 2 * t, 24 + 2 * t, 25 + 2 * t};
            uint32_t w0 = 0, w1 = 0;
            for (int k = 0; k < 4; ++k) {
                w0 |= (uint32_t)((in ? q[e[k]] : 0) ^ 0x80u) << (8 * k);
                w1 |= (uint32_t)((in ? q[e[k + 4]] : 0) ^ 0x80u) << (8 * k);
            }
            words[2 * h] = w0;
            words[2 * h + 1] = w1;
        }
        const int64_t ro = (tau * NJ + j) * 4352;
        if (QG_OK(qg_in(ro + (p * 32 + l) * 16, 16, pack_bytes), st, 302))
            *reinterpret_cast<uint4*>(region + (p * 32 + l) * 16) = make_uint4(words[0], words[1], words[2], words[3]);
        if (l < 16) {
            const int64_t n = tau * 16 + l;
            const bool in = n < N && QG_OK(qg_in((n * NB + b) * 34, 2, canon_bytes), st, 303);
            const uint16_t d = in ? *reinterpret_cast<const uint16_t*>(canon + (n * NB + b) * 34) : (uint16_t)0;
            if (QG_OK(qg_in(ro + 4096 + (p * 16 + l) * 2, 2, pack_bytes), st, 304))
                *reinterpret_cast<uint16_t*>(region + 4096 + (p * 16 + l) * 2) = d;
        }
    }
}

int launch_qpack_q8_0(const void* canon, void* pack, int N, int K, cudaStream_t s)
{
    const int64_t total = (int64_t)((N + 15) / 16) * (K / QK) * 32;
    const int64_t grid = total / 256 + 1 < 65535 ? total / 256 + 1 : 65535;
    qpack_q8_0_kernel<<<(unsigned)grid, 256, 0, s>>>(static_cast<const uint8_t*>(canon), static_cast<uint8_t*>(pack),
                                                     N, K, wait_timeout_counter());
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

// Q4_K (llama.cpp superblock of 256: fp16 d, fp16 dmin, 12 bytes holding
// eight 6-bit scales and eight 6-bit mins, 128 bytes of 4-bit codes; values
// 64c .. 64c+31 are the low nibbles of code bytes 32c .. 32c+31, values
// 64c+32 .. 64c+63 their high nibbles) into the tensor-core pack: per 16-row
// tile and superblock one 2368-byte region = codes [block p][lane 4g + t] 8 B
// (word t of row g's, then of row g + 8's, 16 bytes in the Q4_0 nibble order:
// byte k = value k | value k + 16 << 4 of block p), then [row][p] {scale,
// min}, then [row] {d, dmin} bits.  Rows past N are zeros.  One thread per
// (tile, superblock, row).
__device__ __forceinline__ void q4_k_unpack_scale_min(const uint8_t* s, int j, uint32_t& sc, uint32_t& m)
{
    if (j < 4) {
        sc = s[j] & 63u;
        m = s[j + 4] & 63u;
    } else {
        sc = (s[j + 4] & 15u) | ((uint32_t)(s[j - 4] >> 6) << 4);
        m = (uint32_t)(s[j + 4] >> 4) | ((uint32_t)(s[j] >> 6) << 4);
    }
}

// Q5_K (Q4_K plus qh[32] after the scale bytes: the fifth bit of value i is
// bit i / 32 of qh[i % 32]) into the same layout with, after the codes, a
// [p][row] word of fifth bits (byte k bit s = value k + 4 s of block p);
// region 2880 B.
template <bool FIVE>
__global__ void qpack_q4_k_kernel(const uint8_t* __restrict__ canon, uint8_t* __restrict__ pack, int N, int K,
                                  unsigned int* st)
{
    constexpr int CB = FIVE ? 176 : 144, RB = FIVE ? 2880 : 2368, SCM = FIVE ? 2560 : 2048;
    const int NS = K / QK_K;
    const int64_t T = (N + 15) / 16;
    const int64_t total = T * NS * 16;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(i & 15);
        const int64_t ts = i >> 4;
        const int64_t tau = ts / NS;
        const int sbi = (int)(ts - tau * NS);
        const int64_t n = tau * 16 + r;
        uint8_t* region = pack + (tau * NS + sbi) * RB;
        const int g = r & 7, half = r >> 3;
        // every write below falls in this tile's region, every read in row n's superblock
        if (!QG_OK(qg_in((tau * NS + sbi) * RB, RB, T * NS * RB), st, 311)) continue;
        if (n < N && !QG_OK(qg_in((n * NS + sbi) * CB, CB, (int64_t)N * NS * CB), st, 312)) continue;
        if (n >= N) {
            for (int p = 0; p < 8; ++p) {
                for (int t = 0; t < 4; ++t)
                    *reinterpret_cast<uint32_t*>(region + p * 256 + (4 * g + t) * 8 + 4 * half) = 0u;
                if (FIVE) *reinterpret_cast<uint32_t*>(region + 2048 + (p * 16 + r) * 4) = 0u;
                *reinterpret_cast<uint16_t*>(region + SCM + (r * 8 + p) * 2) = 0;
            }
            *reinterpret_cast<uint32_t*>(region + SCM + 256 + r * 4) = 0u;
            continue;
        }
        const uint8_t* sb = canon + (n * NS + sbi) * CB;
        const uint8_t* qs = sb + (FIVE ? 48 : 16);
        for (int p = 0; p < 8; ++p) {
            const int base = 32 * (p >> 1), shift = 4 * (p & 1);
            for (int t = 0; t < 4; ++t) {
                uint32_t word = 0;
                for (int k = 0; k < 4; ++k) {
                    const int v = 4 * t + k;  // values v and v + 16 of block p
                    const uint32_t lo = (qs[base + v] >> shift) & 15u, hi = (qs[base + v + 16] >> shift) & 15u;
                    word |= (lo | hi << 4) << (8 * k);
                }
                *reinterpret_cast<uint32_t*>(region + p * 256 + (4 * g + t) * 8 + 4 * half) = word;
            }
            if (FIVE) {
                uint32_t hw = 0;
                for (int k = 0; k < 4; ++k)
                    for (int s2 = 0; s2 < 8; ++s2) hw |= (uint32_t)((sb[16 + k + 4 * s2] >> p) & 1) << (8 * k + s2);
                *reinterpret_cast<uint32_t*>(region + 2048 + (p * 16 + r) * 4) = hw;
            }
            uint32_t sc, m;
            q4_k_unpack_scale_min(sb + 4, p, sc, m);
            *reinterpret_cast<uint16_t*>(region + SCM + (r * 8 + p) * 2) = (uint16_t)(sc | m << 8);
        }
        *reinterpret_cast<uint32_t*>(region + SCM + 256 + r * 4) =
            (uint32_t)sb[0] | (uint32_t)sb[1] << 8 | (uint32_t)sb[2] << 16 | (uint32_t)sb[3] << 24;
    }
}

int launch_qpack_q4_k(const void* canon, void* pack, int N, int K, cudaStream_t s)
{
    const int64_t total = (int64_t)((N + 15) / 16) * (K / QK_K) * 16;
    const int64_t grid = total / 256 + 1 < 65535 ? total / 256 + 1 : 65535;
    qpack_q4_k_kernel<false><<<(unsigned)grid, 256, 0, s>>>(static_cast<const uint8_t*>(canon),
                                                            static_cast<uint8_t*>(pack), N, K, wait_timeout_counter());
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

int launch_qpack_q5_k(const void* canon, void* pack, int N, int K, cudaStream_t s)
{
    const int64_t total = (int64_t)((N + 15) / 16) * (K / QK_K) * 16;
    const int64_t grid = total / 256 + 1 < 65535 ? total / 256 + 1 : 65535;
    qpack_q4_k_kernel<true><<<(unsigned)grid, 256, 0, s>>>(static_cast<const uint8_t*>(canon),
                                                           static_cast<uint8_t*>(pack), N, K, wait_timeout_counter());
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

__global__ void qpack_q4_0_kernel(const uint8_t* __restrict__ canon, uint8_t* __restrict__ pack, int N, int K,
                                  unsigned int* st)
{
    const Layout L = make_layout(FMT_Q4_0, N, K);
    const int64_t nblocks = (int64_t)N * L.NB;
    const int64_t total = L.total_bytes();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nblocks;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / L.NB;
        const int b = (int)(i - n * L.NB);
        const uint16_t* src = reinterpret_cast<const uint16_t*>(canon + i * Q4_0_BYTES);  // 2-byte aligned
        uint32_t q[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) q[k] = (uint32_t)src[1 + 2 * k] | ((uint32_t)src[2 + 2 * k] << 16);
        const BlockAddr ad = block_addr(pack, L, n, b);
        if (QG_OK(qg_in(ad.q - pack, 16, total), st, 321))
            *reinterpret_cast<uint4*>(const_cast<uint8_t*>(ad.q)) = make_uint4(q[0], q[1], q[2], q[3]);
        if (QG_OK(qg_in(ad.d - pack, 2, total), st, 322)) *reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(ad.d)) = src[0];
        const int rows = L.rows_in(n / GROUP), c = b / CHUNK, nb = L.nb(c);
        if ((n % GROUP) == 0 && b % CHUNK == 0) {  // zero the group-chunk's pad bytes
            uint8_t* gc = pack + L.chunk_offset(n / GROUP, c);
            for (int p = nb * rows * 18; p < L.chunk_bytes(rows, c); ++p)
                if (QG_OK(qg_in(gc + p - pack, 1, total), st, 323)) gc[p] = 0;
        }
    }
}

__global__ void qpack_q6_k_kernel(const uint8_t* __restrict__ canon, uint8_t* __restrict__ pack, int N, int K,
                                  unsigned int* st)
{
    const Layout L = make_layout(FMT_Q6_K, N, K);
    const int64_t nblocks = (int64_t)N * L.NB;
    const int64_t total = L.total_bytes();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nblocks;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / L.NB;
        const int b = (int)(i - n * L.NB);
        const int64_t sbi = i >> 3;  // superblock index (n * NSB + b / 8)
        const int bb = b & 7;
        const uint8_t* sb = canon + sbi * Q6_K_BYTES;
        // canonical sequential packing: low4(q_v) = nibble (v & 1) of ql[v >> 1],
        // high2(q_v) = bits 2 (v & 3) of qh[v >> 2]; this block's values are
        // v = 32 bb .. 32 bb + 31 of the superblock.
        uint8_t q[32];
#pragma unroll
        for (int v = 0; v < 32; ++v) {
            const int gv = 32 * bb + v;
            const int lo = (sb[gv >> 1] >> (4 * (gv & 1))) & 0x0F;
            const int hi = (sb[128 + (gv >> 2)] >> (2 * (gv & 3))) & 0x03;
            q[v] = (uint8_t)(lo | (hi << 4));
        }
        // P[16]: byte t = q_t | high2(q_{16+t}) << 6; Q[8]: byte u =
        // low4(q_{16+u}) | low4(q_{24+u}) << 4 (q6_k_unpack reads them back)
        uint32_t wl[4] = {0, 0, 0, 0};
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            const uint32_t byte = (uint32_t)q[t] | ((uint32_t)(q[t + 16] >> 4) << 6);
            wl[t >> 2] |= byte << (8 * (t & 3));
        }
        uint32_t wh[2] = {0, 0};
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint32_t byte = (uint32_t)(q[16 + u] & 0x0F) | ((uint32_t)(q[24 + u] & 0x0F) << 4);
            wh[u >> 2] |= byte << (8 * (u & 3));
        }
        const BlockAddr ad = block_addr(pack, L, n, b);
        if (QG_OK(qg_in(ad.q - pack, 16, total) && qg_in(ad.qh - pack, 8, total) && qg_in(ad.sc - pack, 2, total) &&
                      qg_in(ad.d - pack, 2, total),
                  st, 331)) {
            *reinterpret_cast<uint4*>(const_cast<uint8_t*>(ad.q)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
            *reinterpret_cast<uint2*>(const_cast<uint8_t*>(ad.qh)) = make_uint2(wh[0], wh[1]);
            *reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(ad.sc)) =
                (uint16_t)sb[192 + 2 * bb] | ((uint16_t)sb[192 + 2 * bb + 1] << 8);
            if (bb == 0)
                *reinterpret_cast<uint16_t*>(const_cast<uint8_t*>(ad.d)) = (uint16_t)sb[208] | ((uint16_t)sb[209] << 8);
        }
        const int rows = L.rows_in(n / GROUP), c = b / CHUNK, nb = L.nb(c);
        if ((n % GROUP) == 0 && b % CHUNK == 0) {  // zero the scale part's pad bytes
            uint8_t* dq = pack + L.chunk_offset(n / GROUP, c) + rows * nb * 26;
            for (int p = rows * (nb / 8) * 2; p < pad16(rows * (nb / 8) * 2); ++p)
                if (QG_OK(qg_in(dq + p - pack, 1, total), st, 332)) dq[p] = 0;
        }
    }
}

static int grid_for(int64_t n, int threads, int sms)
{
    int64_t g = (n + threads - 1) / threads;
    const int64_t cap = (int64_t)sms * 16;
    return (int)(g < 1 ? 1 : (g > cap ? cap : g));
}

int launch_qpack_q4_0(const void* canon, void* pack, int N, int K, cudaStream_t s)
{
    const DeviceInfo di = device_info();
    if (di.sms <= 0) return QGEMV_CUDA_ERROR;
    const int64_t nblocks = (int64_t)N * (K / QK);
    qpack_q4_0_kernel<<<grid_for(nblocks, 256, di.sms), 256, 0, s>>>(static_cast<const uint8_t*>(canon),
                                                                     static_cast<uint8_t*>(pack), N, K,
                                                                     wait_timeout_counter());
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

int launch_qpack_q6_k(const void* canon, void* pack, int N, int K, cudaStream_t s)
{
    const DeviceInfo di = device_info();
    if (di.sms <= 0) return QGEMV_CUDA_ERROR;
    const int64_t nblocks = (int64_t)N * (K / QK);
    qpack_q6_k_kernel<<<grid_for(nblocks, 256, di.sms), 256, 0, s>>>(static_cast<const uint8_t*>(canon),
                                                                     static_cast<uint8_t*>(pack), N, K,
                                                                     wait_timeout_counter());
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

// ---------------------------------------------------------------------------
// argmax_f32_rows: the separate argmax of the unfused LM-head path ("Q6_K M=6
// fused DFlash top-1 production record", Why this was slow), with the same
// lowest-ID tie contract as the fused reducer (Exactness and safety
// contracts, item 3).  Cross-CTA reduction: 64-bit atomicMax on the
// order-preserving key, then the last CTA to finish writes the ids and resets
// the workspace.
// ---------------------------------------------------------------------------

constexpr int ARGMAX_THREADS = 256;

template <int M>
__global__ void __launch_bounds__(ARGMAX_THREADS) argmax_rows_kernel(const float* __restrict__ y, int64_t ldy,
                                                                     int32_t* __restrict__ ids, Top1Workspace* ws,
                                                                     int N, unsigned int* st)
{
    __shared__ unsigned long long s_red[ARGMAX_THREADS / 32][M];
    __shared__ int s_last;
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long k[M];
#pragma unroll
    for (int m = 0; m < M; ++m) k[m] = 0ull;
    const bool vec4 = ((reinterpret_cast<uintptr_t>(y) | ((uintptr_t)ldy * 4)) & 15u) == 0;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t extent = (int64_t)(M - 1) * ldy + N;  // elements of y read
    if (vec4) {
        const int64_t n4 = N / 4;
        for (int64_t q = tid; q < n4; q += nthreads) {
            float4 v[M];
#pragma unroll
            for (int m = 0; m < M; ++m)
                v[m] = QG_OK(qg_in((int64_t)m * ldy + 4 * q, 4, extent), st, 401)
                           ? __ldg(reinterpret_cast<const float4*>(y + (int64_t)m * ldy) + q)
                           : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const int n = (int)(4 * q);
                unsigned long long c;
                c = top1_key(v[m].x, n);
                k[m] = c > k[m] ? c : k[m];
                c = top1_key(v[m].y, n + 1);
                k[m] = c > k[m] ? c : k[m];
                c = top1_key(v[m].z, n + 2);
                k[m] = c > k[m] ? c : k[m];
                c = top1_key(v[m].w, n + 3);
                k[m] = c > k[m] ? c : k[m];
            }
        }
        for (int64_t n = 4 * n4 + tid; n < N; n += nthreads) {
#pragma unroll
            for (int m = 0; m < M; ++m) {
                if (!QG_OK(qg_in((int64_t)m * ldy + n, 1, extent), st, 402)) continue;
                const unsigned long long c = top1_key(__ldg(y + (int64_t)m * ldy + n), (int)n);
                k[m] = c > k[m] ? c : k[m];
            }
        }
    } else {
        for (int64_t n = tid; n < N; n += nthreads) {
#pragma unroll
            for (int m = 0; m < M; ++m) {
                if (!QG_OK(qg_in((int64_t)m * ldy + n, 1, extent), st, 402)) continue;
                const unsigned long long c = top1_key(__ldg(y + (int64_t)m * ldy + n), (int)n);
                k[m] = c > k[m] ? c : k[m];
            }
        }
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const unsigned long long w = warp_max_u64(k[m]);
        if (lane == 0) s_red[warp][m] = w;
    }
    __syncthreads();
    if (threadIdx.x < M) {
        unsigned long long b = 0ull;
        for (int w = 0; w < ARGMAX_THREADS / 32; ++w) b = s_red[w][threadIdx.x] > b ? s_red[w][threadIdx.x] : b;
        atomicMax(&ws->keys[threadIdx.x], b);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = atomicAdd(&ws->done, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        if (threadIdx.x < M) ids[threadIdx.x] = top1_key_to_id(atomicExch(&ws->keys[threadIdx.x], 0ull));
        if (threadIdx.x == 0) atomicExch(&ws->done, 0u);
    }
}

template <int M>
static cudaError_t launch_argmax_m(const float* y, int64_t ldy, int32_t* ids, Top1Workspace* ws, int N, int grid,
                                   cudaStream_t s)
{
    return launch_pdl(argmax_rows_kernel<M>, dim3(grid), dim3(ARGMAX_THREADS), 0, s, y, ldy, ids, ws, N,
                      wait_timeout_counter());
}

int launch_argmax_rows(const float* y, int64_t ldy, int32_t* ids, Top1Workspace* ws, int M, int N, cudaStream_t s)
{
    const DeviceInfo di = device_info();
    if (di.sms <= 0) return QGEMV_CUDA_ERROR;
    int grid = (int)(((int64_t)N + ARGMAX_THREADS * 4 - 1) / (ARGMAX_THREADS * 4));
    if (grid > di.sms * 2) grid = di.sms * 2;
    if (grid < 1) grid = 1;
    cudaError_t e = cudaSuccess;
    switch (M) {
#define QGEMV_ARGMAX_CASE(m) \
    case m: e = launch_argmax_m<m>(y, ldy, ids, ws, N, grid, s); break;
    QGEMV_ARGMAX_CASE(1) QGEMV_ARGMAX_CASE(2) QGEMV_ARGMAX_CASE(3) QGEMV_ARGMAX_CASE(4) QGEMV_ARGMAX_CASE(5)
    QGEMV_ARGMAX_CASE(6) QGEMV_ARGMAX_CASE(7) QGEMV_ARGMAX_CASE(8) QGEMV_ARGMAX_CASE(9) QGEMV_ARGMAX_CASE(10)
    QGEMV_ARGMAX_CASE(11) QGEMV_ARGMAX_CASE(12) QGEMV_ARGMAX_CASE(13) QGEMV_ARGMAX_CASE(14)
    QGEMV_ARGMAX_CASE(15) QGEMV_ARGMAX_CASE(16) QGEMV_ARGMAX_CASE(17)
#undef QGEMV_ARGMAX_CASE
    default: return QGEMV_UNSUPPORTED_SHAPE;
    }
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

// ---------------------------------------------------------------------------
// Integer block dots, for checking them bit for bit: out[m][n][b] is the
// exact int32 dot of weight block (n, b) with activation block (m, b), made by
// the same staging, unpacking and dot routines as the MMVQ kernels.
// ---------------------------------------------------------------------------

template <int FMT>
__global__ void block_dots_kernel(const void* __restrict__ w_pack, const uint8_t* __restrict__ xq,
                                  int32_t* __restrict__ out, int M, int NB, int N, unsigned int* st)
{
    const int64_t total = (int64_t)M * N * NB;
    const Layout L = make_layout(FMT, N, NB * QK);
    const int64_t wbytes = L.total_bytes();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int b = (int)(i % NB);
        const int64_t mn = i / NB;
        const int n = (int)(mn % N), m = (int)(mn / N);
        uint4 lo, hi;
        uint2 meta;
        if (!QG_OK(qg_in(((int64_t)m * NB + b) * Q8_1_BYTES, Q8_1_BYTES, (int64_t)M * NB * Q8_1_BYTES), st, 501))
            continue;
        act_from_q8_1<FMT>(xq + ((int64_t)m * NB + b) * Q8_1_BYTES, lo, hi, meta);
        uint32_t w[8];
        const BlockAddr ad = block_addr(w_pack, L, n, b);
        const uint8_t* w0 = static_cast<const uint8_t*>(w_pack);
        if (!QG_OK(qg_in(ad.q - w0, 16, wbytes) && (FMT == FMT_Q4_0 || (qg_in(ad.qh - w0, 8, wbytes) &&
                                                                      qg_in(ad.sc - w0, 2, wbytes))),
                   st, 502))
            continue;
        if (FMT == FMT_Q4_0) {
            q4_0_unpack(*reinterpret_cast<const uint4*>(ad.q), w);
            out[i] = q4_0_dot(w, lo, hi, (int)meta.y);
        } else {
            q6_k_unpack(*reinterpret_cast<const uint4*>(ad.q), *reinterpret_cast<const uint2*>(ad.qh), w);
            out[i] = q6_k_dot(w, lo, hi, meta.y, *reinterpret_cast<const uint16_t*>(ad.sc)) >> 2;  // 4 J -> J, exact
        }
    }
}

int launch_block_dots(int fmt, const void* w_pack, const void* xq, int32_t* out, int M, int K, int N, cudaStream_t s)
{
    const DeviceInfo di = device_info();
    if (di.sms <= 0) return QGEMV_CUDA_ERROR;
    const int NB = K / QK;
    const int64_t total = (int64_t)M * N * NB;
    const int grid = grid_for(total, 256, di.sms);
    if (fmt == FMT_Q4_0)
        block_dots_kernel<FMT_Q4_0><<<grid, 256, 0, s>>>(w_pack, static_cast<const uint8_t*>(xq), out, M, NB, N,
                                                         wait_timeout_counter());
    else
        block_dots_kernel<FMT_Q6_K><<<grid, 256, 0, s>>>(w_pack, static_cast<const uint8_t*>(xq), out, M, NB, N,
                                                         wait_timeout_counter());
    return cudaGetLastError() == cudaSuccess ? QGEMV_OK : QGEMV_CUDA_ERROR;
}

}  // namespace qgemv
