// FP8 input preparation for sm_103a (FlashAttention from Scratch, sec. 10.3
// "Treat FP8 as a second lesson"; FlashAttention 1-4, FA3 item 3 "FP8 with
// block quantization and incoherent processing").
//
// Q and K rows are multiplied by the same orthogonal matrix
// M = diag(signs) H / sqrt(128) -- a fast Walsh-Hadamard transform of the
// sign-flipped row, O(d log d) per row -- which leaves Q K^T unchanged and
// spreads outlier coordinates over the whole row; then every 128-row tile of
// a (batch, head) slice is quantised to e4m3 with its own scale
// amax(tile) / 448.  V keeps its coordinates (a rotation would have to be
// undone on O), gets one scale per (batch, KV head) slice, and is stored
// transposed ([d][key]) so that it is a K-major operand of the P.V MMA.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_fp8.h"

namespace fa {

namespace {

constexpr float kE4m3Max = 448.f;

// Two fp32 values to two e4m3 codes, round to nearest even, saturating;
// `lo` ends in the low byte (the lower address).
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float block_max128(float x, float* red)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
    __syncthreads();
    const float m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    return m;
}

// One CTA (128 threads) per 128-row tile of Q or K; thread = row.
__global__ void __launch_bounds__(128) fa_fp8_qk_kernel(const Fp8PrepParams p)
{
    __shared__ float sgn[128];
    __shared__ float red[4];
    sgn[threadIdx.x] = p.signs[threadIdx.x];
    const int nq_blocks = p.B * p.Hq * p.nq;
    int blk = blockIdx.x;
    const bool is_q = blk < nq_blocks;
    if (!is_q) blk -= nq_blocks;
    const int per = is_q ? p.nq : p.nk;
    const int slice = blk / per, tile = blk - slice * per;
    const int L = is_q ? p.Lq : p.Lk;
    const uint16_t* src = is_q ? p.q : p.k;
    uint8_t* dst = is_q ? p.qc : p.kc;
    const int row = tile * kFp8Tile + threadIdx.x;
    const bool valid = row < L;
    __syncthreads();
    float x[128];
    if (valid) {
        const uint4* s4 = reinterpret_cast<const uint4*>(src + ((long long)slice * L + row) * 128);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const uint4 u = __ldg(s4 + c);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[8 * c + 2 * e] = __uint_as_float(w[e] << 16) * sgn[8 * c + 2 * e];
                x[8 * c + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u) * sgn[8 * c + 2 * e + 1];
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 128; ++i) x[i] = 0.f;
    }
    // Walsh-Hadamard butterflies, natural (Sylvester) order, then 1/sqrt(128)
#pragma unroll
    for (int st = 0; st < 7; ++st) {
        const int h = 1 << st;
#pragma unroll
        for (int i = 0; i < 64; ++i) {  // the 64 butterflies of stage st: pairs (j, j + h)
            const int j = ((i >> st) << (st + 1)) | (i & (h - 1));
            const float a = x[j], b = x[j + h];
            x[j] = a + b;
            x[j + h] = a - b;
        }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 128; ++i) {
        x[i] *= 0.08838834764831845f;  // 1 / sqrt(128)
        amax = fmaxf(amax, fabsf(x[i]));
    }
    amax = block_max128(amax, red);
    const float scale = amax > 0.f ? amax / kE4m3Max : 1.f;
    if (threadIdx.x == 0) (is_q ? p.sq : p.sk)[blk] = scale;
    if (valid) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + ((long long)slice * L + row) * 128);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = 16 * c + 4 * e;
                w[e] = (uint32_t)e4m3x2(__fdiv_rn(x[i], scale), __fdiv_rn(x[i + 1], scale)) |
                       ((uint32_t)e4m3x2(__fdiv_rn(x[i + 2], scale), __fdiv_rn(x[i + 3], scale)) << 16);
            }
            d4[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// amax of every V slice: CTAs stride over a slice's elements, atomicMax on the
// (non-negative) float bits.
__global__ void __launch_bounds__(256) fa_fp8_vmax_kernel(const Fp8PrepParams p, int ctas_per_slice)
{
    __shared__ float red[8];
    const int slice = blockIdx.x / ctas_per_slice, part = blockIdx.x - slice * ctas_per_slice;
    const long long n8 = (long long)p.Lk * 128 / 8;  // uint4 per slice
    const uint4* s4 = reinterpret_cast<const uint4*>(p.v + (long long)slice * p.Lk * 128);
    float m = 0.f;
    for (long long i = (long long)part * 256 + threadIdx.x; i < n8; i += (long long)ctas_per_slice * 256) {
        const uint4 u = __ldg(s4 + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[e] << 16)), fabsf(__uint_as_float(w[e] & 0xffff0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = red[0];
        for (int w = 1; w < 8; ++w) b = fmaxf(b, red[w]);
        atomicMax(p.vmax + slice, __float_as_uint(b));
    }
}

// One CTA per 128-key tile of a V slice: quantise with the slice scale and
// write the tile transposed, [d][key].
__global__ void __launch_bounds__(128) fa_fp8_v_kernel(const Fp8PrepParams p)
{
    __shared__ uint8_t tile[128][144];  // [key][d], rows padded against bank conflicts
    const int ntile = p.Lk_pad / kFp8Tile;
    const int slice = blockIdx.x / ntile, t = blockIdx.x - slice * ntile;
    const float amax = __uint_as_float(p.vmax[slice]);
    const float scale = amax > 0.f ? amax / kE4m3Max : 1.f;
    if (t == 0 && threadIdx.x == 0) p.sv[slice] = scale;
    const int key = t * kFp8Tile + threadIdx.x;
    uint32_t* trow = reinterpret_cast<uint32_t*>(&tile[threadIdx.x][0]);
    if (key < p.Lk) {
        const uint4* s4 = reinterpret_cast<const uint4*>(p.v + ((long long)slice * p.Lk + key) * 128);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const uint4 u = __ldg(s4 + c);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
            const float f0 = __fdiv_rn(__uint_as_float(w[0] << 16), scale);
            const float f1 = __fdiv_rn(__uint_as_float(w[0] & 0xffff0000u), scale);
            const float f2 = __fdiv_rn(__uint_as_float(w[1] << 16), scale);
            const float f3 = __fdiv_rn(__uint_as_float(w[1] & 0xffff0000u), scale);
            const float f4 = __fdiv_rn(__uint_as_float(w[2] << 16), scale);
            const float f5 = __fdiv_rn(__uint_as_float(w[2] & 0xffff0000u), scale);
            const float f6 = __fdiv_rn(__uint_as_float(w[3] << 16), scale);
            const float f7 = __fdiv_rn(__uint_as_float(w[3] & 0xffff0000u), scale);
            trow[2 * c] = (uint32_t)e4m3x2(f0, f1) | ((uint32_t)e4m3x2(f2, f3) << 16);
            trow[2 * c + 1] = (uint32_t)e4m3x2(f4, f5) | ((uint32_t)e4m3x2(f6, f7) << 16);
        }
    } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) trow[c] = 0u;
    }
    __syncthreads();
    // thread = d: gather the tile's 128 keys of dimension d
    const int d = threadIdx.x;
    uint32_t w[32];
#pragma unroll
    for (int c = 0; c < 32; ++c)
        w[c] = (uint32_t)tile[4 * c][d] | ((uint32_t)tile[4 * c + 1][d] << 8) | ((uint32_t)tile[4 * c + 2][d] << 16) |
               ((uint32_t)tile[4 * c + 3][d] << 24);
    uint4* d4 = reinterpret_cast<uint4*>(p.vt + ((long long)slice * 128 + d) * p.Lk_pad + t * kFp8Tile);
#pragma unroll
    for (int c = 0; c < 8; ++c) d4[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}

}  // namespace

cudaError_t launch_fp8_prepare(const Fp8PrepParams& p, cudaStream_t stream)
{
    const int qk_blocks = p.B * p.Hq * p.nq + p.B * p.Hkv * p.nk;
    fa_fp8_qk_kernel<<<qk_blocks, 128, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int slices = p.B * p.Hkv;
    const int per = (int)((((long long)p.Lk * 16) + 255) / 256 < 64 ? (((long long)p.Lk * 16) + 255) / 256 : 64);
    fa_fp8_vmax_kernel<<<slices * (per > 0 ? per : 1), 256, 0, stream>>>(p, per > 0 ? per : 1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    fa_fp8_v_kernel<<<slices * (p.Lk_pad / kFp8Tile), 128, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace fa
