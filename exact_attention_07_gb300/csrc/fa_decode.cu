// Split-KV decode forward for sm_103a: a partial kernel per key-range
// partition and an LSE-weighted merge (FlashAttention from Scratch, sec. 9.1
// "Split the long dimension that remains", sec. 4.3 "Merge independently
// computed partitions", sec. 9.2 "GQA changes the reuse opportunity").
//
// Decode reads every K and V element once and does 2 * R * D multiply-adds per
// key (R = query rows that share the KV head), a few FLOP per byte: the work
// is bound by HBM bandwidth, not by the tensor cores.  So the kernels stream
// K/V through shared memory with TMA and do the arithmetic on the FP32 pipes;
// what matters is keeping enough bytes in flight (a 3- or 4-stage ring per
// CTA, two CTAs per SM) and keeping shared-memory traffic conflict free.
//
// One partial CTA owns one (batch, KV head, partition) and all R query rows
// of the group, so each K/V byte is read from HBM once for all of them.
// Per 64-key tile:
//   1. S phase: warp (key half, dimension quarter) -- each lane takes one
//      key and a quarter of D, for every row; partial dot products go to
//      shared memory.  K chunks are read with the tile's 128-byte swizzle.
//   2. softmax phase: one warp per row adds the four quarters, masks, and
//      runs the online-softmax update (running maximum m, running sum l,
//      rescale factor alpha = 2^(m_old - m_new)).
//   3. P.V phase: each lane owns 8 output dimensions of a few rows and every
//      eighth key of the tile; the accumulators are rescaled by alpha and
//      updated with p * V.  The eight warps' partial sums are added once at
//      the end.
// The partition's output is normalised, O_s = A / l, with the base-2
// log-sum-exp m + log2 l beside it; a single-partition launch writes the
// final O and natural-log LSE directly.
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa_decode.h"
#include "ptx_sm103.cuh"

namespace fa {

template <int D>
struct DecCfg {
    static constexpr int CH = D / 8;                      // 16-byte chunks of one key row
    static constexpr int HALVES = D / 64;                 // 128-byte TMA boxes of one key row
    static constexpr int BOX_BYTES = kDecKeys * 128;      // one 64-key x 64-dim box
    static constexpr int TILE_BYTES = HALVES * BOX_BYTES;  // K (or V) of one tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;    // K and V
    static constexpr int NS = D == 128 ? 3 : 4;           // ring stages
    static constexpr int RG = 32 / CH;                    // lane groups over rows in P.V
    static constexpr int CPQ = CH / 4;                    // chunks per dimension quarter in S
};

// Shared-memory layout after the 1024-byte-aligned ring, in floats.
template <int D, int RMAX>
struct DecSmem {
    static constexpr int RING = DecCfg<D>::NS * DecCfg<D>::STAGE_BYTES;
    static constexpr int Q = 0;                         // [RMAX][D] query rows, scaled to log2 units
    static constexpr int PART = Q + RMAX * D;           // [4][RMAX][64] dot-product quarters
    static constexpr int P = PART + 4 * RMAX * kDecKeys;  // [64][RMAX] probabilities, P.V order
    static constexpr int ALPHA = P + kDecKeys * RMAX;   // [RMAX]
    static constexpr int M = ALPHA + RMAX;              // [RMAX] final running maximum
    static constexpr int L = M + RMAX;                  // [RMAX] final running sum
    static constexpr int FLOATS = (L + RMAX + 3) & ~3;
    static constexpr int BARS = RING + FLOATS * 4;      // byte offset of the mbarriers
    static constexpr int BYTES = BARS + DecCfg<D>::NS * 8 + 16;
    static constexpr int DYNAMIC = BYTES + 1024;        // + alignment slack
    static_assert(8 * RMAX * D * 4 <= RING, "warp reduction buffer must fit in the ring");
};

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// Eight bf16 values (one 16-byte chunk) to fp32; bf16 is the high half of fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8])
{
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xffff0000u);
    f[4] = __uint_as_float(u.z << 16);
    f[5] = __uint_as_float(u.z & 0xffff0000u);
    f[6] = __uint_as_float(u.w << 16);
    f[7] = __uint_as_float(u.w & 0xffff0000u);
}

// 16 bytes of fp32 from shared memory as two packed pairs.
__device__ __forceinline__ void lds128_f2(uint32_t addr, uint64_t& a, uint64_t& b)
{
    asm volatile("ld.shared.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "r"(addr));
}

// Eight bf16 values to four packed fp32 pairs (dimensions 2i, 2i + 1).
__device__ __forceinline__ void bf16x8_to_f2(const uint4& u, uint64_t (&f)[4])
{
    f[0] = f2_pack(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u));
    f[1] = f2_pack(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    f[2] = f2_pack(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u));
    f[3] = f2_pack(__uint_as_float(u.w << 16), __uint_as_float(u.w & 0xffff0000u));
}

// Byte offset of 16-byte chunk c of key row `key` inside a tile that TMA wrote
// with the 128-byte swizzle: chunk index XOR (row mod 8) within each 128-byte
// row, boxes of 64 dimensions back to back.
template <int D>
__device__ __forceinline__ uint32_t tile_chunk(int key, int c)
{
    return (uint32_t)((c >> 3) * DecCfg<D>::BOX_BYTES + key * 128 + (((c & 7) ^ (key & 7)) << 4));
}

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// ------------------------------------------------------------------ partial kernel

// Thread 0 only: arm the stage's barrier and load K and V of tile t.
template <int D>
__device__ __forceinline__ void dec_issue(uint32_t ring, uint32_t bars, const CUtensorMap* tk,
                                          const CUtensorMap* tv, int t, int key0, int bh)
{
    using C = DecCfg<D>;
    const int st = t % C::NS;
    const uint32_t stage = ring + st * C::STAGE_BYTES;
    const uint32_t bar = bars + st * 8;
    mbar_arrive_expect_tx(bar, C::STAGE_BYTES);
#pragma unroll
    for (int h = 0; h < C::HALVES; ++h) {
        tma_load_3d(stage + h * C::BOX_BYTES, tk, bar, 64 * h, key0, bh);
        tma_load_3d(stage + C::TILE_BYTES + h * C::BOX_BYTES, tv, bar, 64 * h, key0, bh);
    }
}

// CTAs per SM that the shared memory of one instantiation allows (228 KiB
// per SM, 1 KiB of it reserved per CTA); the register budget follows it.
template <int D, int RPT>
constexpr int dec_min_blocks()
{
    return 2 * (DecSmem<D, DecCfg<D>::RG * RPT>::DYNAMIC + 1024) <= 233472 ? 2 : 1;
}

template <int D, int RPT>
__global__ void __launch_bounds__(kDecThreads, dec_min_blocks<D, RPT>())
    fa_decode_partial_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                             const DecodeParams p)
{
    using C = DecCfg<D>;
    constexpr int RMAX = C::RG * RPT;
    using S = DecSmem<D, RMAX>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t ring = (raw + 1023u) & ~1023u;
    uint8_t* sbase = smem_raw + (ring - raw);
    float* fs = reinterpret_cast<float*>(sbase + S::RING);
    float* q_s = fs + S::Q;
    float* part_s = fs + S::PART;
    float* p_s = fs + S::P;
    float* alpha_s = fs + S::ALPHA;
    float* m_s = fs + S::M;
    float* l_s = fs + S::L;
    const uint32_t bars = ring + S::BARS;
    const uint32_t q_u32 = ring + S::RING + S::Q * 4;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sbase + S::BARS + C::NS * 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = (int)(blockIdx.x % (unsigned)p.num_splits);
    const int bh = (int)(blockIdx.x / (unsigned)p.num_splits);  // b * Hkv + kv head
    const int b = bh / p.Hkv, hkv = bh - b * p.Hkv;
    const int t0 = split * p.tiles_per_split;
    const int ntiles = min(p.num_tiles - t0, p.tiles_per_split);
    // the R query rows of this KV head are contiguous: heads hkv*group .. +group-1, Lq rows each
    const long long row0 = ((long long)b * p.Hq + (long long)hkv * p.group) * p.Lq;
    const WaitFailure wf{p.err, p.diag};

    if (tid == 0) {
        for (int s = 0; s < C::NS; ++s) mbar_init(bars + s * 8, 1);
        *abort_flag = 0;
        mbar_init_fence();
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
    }
    // query rows to fp32, pre-scaled so that dot products come out in log2 units
    {
        const uint4* qg = reinterpret_cast<const uint4*>(p.q + row0 * D);
        for (int i = tid; i < RMAX * (D / 8); i += kDecThreads) {
            float f[8];
            if (i / (D / 8) < p.R) {
                bf16x8_to_f32(__ldg(qg + i), f);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = 0.f;
            }
            float4* dst = reinterpret_cast<float4*>(q_s + i * 8);
            dst[0] = make_float4(f[0] * p.scale_log2, f[1] * p.scale_log2, f[2] * p.scale_log2, f[3] * p.scale_log2);
            dst[1] = make_float4(f[4] * p.scale_log2, f[5] * p.scale_log2, f[6] * p.scale_log2, f[7] * p.scale_log2);
        }
        for (int i = tid; i < kDecKeys * RMAX; i += kDecThreads) p_s[i] = 0.f;
        if (tid < RMAX) alpha_s[tid] = 1.f;
    }
    __syncthreads();

    int n_issued = 0;
    bool armed0 = true;
    if (tid == 0) {
        const int pre = min(C::NS, ntiles);
        for (int t = 0; t < pre; ++t) {
            if (t == 0 && p.fault == 1) {
                armed0 = false;  // test hook: tile 0 never arrives
            } else {
                dec_issue<D>(ring, bars, &tmK, &tmV, t, (t0 + t) * kDecKeys, bh);
            }
        }
        n_issued = pre;
    }

    // online-softmax state of rows warp and warp + 8 (identical in every lane)
    float m_row[2] = {-INFINITY, -INFINITY};
    float l_row[2] = {0.f, 0.f};  // per-lane share of the running sum
    uint64_t acc[RPT][4];  // packed pairs: dimensions (2e, 2e + 1) of the lane's chunk
#pragma unroll
    for (int u = 0; u < RPT; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[u][e] = 0ull;
    const int c_pv = lane % C::CH, rg = lane / C::CH;
    const int causal_off = p.Lk - p.Lq;

    bool failed = false;
    int j = 0;
    for (; j < ntiles; ++j) {
        const int st = j % C::NS;
        const uint32_t stage = ring + st * C::STAGE_BYTES;
        const bool ok = mbar_wait(bars + st * 8, (uint32_t)((j / C::NS) & 1), abort_flag, wf, 40, j);

        // ---- S phase: lane = key, warp = (key half, dimension quarter); rows
        // in passes of at most 8 to bound the live registers.  Packed fp32
        // pairs: even and odd dimensions accumulate separately, then add.
        {
            const int key = (warp >> 2) * 32 + lane, qq = warp & 3;
            constexpr int RB = RMAX < 8 ? RMAX : 8;
#pragma unroll
            for (int rb = 0; rb < RMAX; rb += RB) {
                uint64_t s2[RB];
#pragma unroll
                for (int r = 0; r < RB; ++r) s2[r] = 0ull;
#pragma unroll
                for (int ci = 0; ci < C::CPQ; ++ci) {
                    const int c = qq * C::CPQ + ci;
                    uint64_t k2[4];
                    bf16x8_to_f2(lds128(stage + tile_chunk<D>(key, c)), k2);
#pragma unroll
                    for (int r = 0; r < RB; ++r) {
                        const uint32_t qa = q_u32 + (uint32_t)(((rb + r) * D + c * 8) * 4);
                        uint64_t q0, q1, q2, q3;
                        lds128_f2(qa, q0, q1);
                        lds128_f2(qa + 16, q2, q3);
                        uint64_t x = s2[r];
                        x = f2_fma(q0, k2[0], x);
                        x = f2_fma(q1, k2[1], x);
                        x = f2_fma(q2, k2[2], x);
                        x = f2_fma(q3, k2[3], x);
                        s2[r] = x;
                    }
                }
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    float lo, hi;
                    f2_unpack(s2[r], lo, hi);
                    part_s[(qq * RMAX + rb + r) * kDecKeys + key] = lo + hi;
                }
            }
        }
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        // every thread is past P.V of tile j - 1: its stage can be refilled
        if (tid == 0 && j >= 1 && j - 1 + C::NS < ntiles) {
            const int t = j - 1 + C::NS;
            dec_issue<D>(ring, bars, &tmK, &tmV, t, (t0 + t) * kDecKeys, bh);
            n_issued = t + 1;
        }

        // ---- softmax phase: warp w updates rows w and w + 8
        const int key_base = (t0 + j) * kDecKeys;
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
            const int r = warp + 8 * ri;
            if (r < p.R) {
                const int qpos = r % p.Lq;
                // last key this row may see (bottom-right causal alignment, and the padding at Lk)
                const int lim = p.causal ? min(p.Lk - 1, qpos + causal_off) : p.Lk - 1;
                float sv[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = lane + 32 * e;
                    const float x = part_s[(0 * RMAX + r) * kDecKeys + key] + part_s[(1 * RMAX + r) * kDecKeys + key] +
                                    part_s[(2 * RMAX + r) * kDecKeys + key] + part_s[(3 * RMAX + r) * kDecKeys + key];
                    sv[e] = (key_base + key <= lim) ? x : -INFINITY;
                }
                const float mn = fmaxf(m_row[ri], warp_max(fmaxf(sv[0], sv[1])));
                float alpha = 1.f, p0 = 0.f, p1 = 0.f;
                if (mn != -INFINITY) {  // a row with no allowed key so far keeps the empty state
                    alpha = ex2_approx(m_row[ri] - mn);
                    p0 = ex2_approx(sv[0] - mn);
                    p1 = ex2_approx(sv[1] - mn);
                }
                l_row[ri] = l_row[ri] * alpha + (p0 + p1);
                m_row[ri] = mn;
                const int pofs = (r % C::RG) * RPT + r / C::RG;
                p_s[lane * RMAX + pofs] = p0;
                p_s[(lane + 32) * RMAX + pofs] = p1;
                if (lane == 0) alpha_s[r] = alpha;
            }
        }
        __syncthreads();

        // ---- P.V phase: lane = (8-dimension chunk, row group), warp = every
        // eighth key; accumulators are packed pairs of adjacent dimensions
        {
#pragma unroll
            for (int u = 0; u < RPT; ++u) {
                const float a = alpha_s[rg + C::RG * u];
                const uint64_t a2 = f2_pack(a, a);
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[u][e] = f2_mul(acc[u][e], a2);
            }
            const uint32_t vtile = stage + C::TILE_BYTES;
#pragma unroll(RPT >= 4 ? 2 : 8)
            for (int i = 0; i < kDecKeys / 8; ++i) {
                const int key = warp + 8 * i;
                uint64_t v2[4];
                bf16x8_to_f2(lds128(vtile + tile_chunk<D>(key, c_pv)), v2);
                float pr[RPT];
                const float* pp = p_s + key * RMAX + rg * RPT;
                if constexpr (RPT == 1) {
                    pr[0] = pp[0];
                } else if constexpr (RPT == 2) {
                    const float2 t = *reinterpret_cast<const float2*>(pp);
                    pr[0] = t.x;
                    pr[1] = t.y;
                } else {
#pragma unroll
                    for (int u4 = 0; u4 < RPT / 4; ++u4) {
                        const float4 t = *reinterpret_cast<const float4*>(pp + 4 * u4);
                        pr[4 * u4 + 0] = t.x;
                        pr[4 * u4 + 1] = t.y;
                        pr[4 * u4 + 2] = t.z;
                        pr[4 * u4 + 3] = t.w;
                    }
                }
#pragma unroll
                for (int u = 0; u < RPT; ++u) {
                    const uint64_t p2 = f2_pack(pr[u], pr[u]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[u][e] = f2_fma(p2, v2[e], acc[u][e]);
                }
            }
        }
    }

    if (failed) {
        // retire: copies already in flight must land before the CTA's shared
        // memory is released; the tile that never arrived is given up after
        // the wait limit
        if (tid == 0) {
            for (int t = j; t < n_issued; ++t) {
                if (t == 0 && !armed0) continue;
                mbar_settle(bars + (t % C::NS) * 8, (uint32_t)((t / C::NS) & 1), wf, 41);
            }
        }
        __syncthreads();
        return;
    }

    // ---- combine the eight warps' key subsets (the ring is free now)
    __syncthreads();
    float* red = reinterpret_cast<float*>(sbase);  // [8][RMAX][D]
#pragma unroll
    for (int u = 0; u < RPT; ++u) {
        float f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) f2_unpack(acc[u][e], f[2 * e], f[2 * e + 1]);
        float4* dst = reinterpret_cast<float4*>(red + (warp * RMAX + rg + C::RG * u) * D + c_pv * 8);
        dst[0] = make_float4(f[0], f[1], f[2], f[3]);
        dst[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
        const int r = warp + 8 * ri;
        if (r < p.R) {
            const float l = warp_sum(l_row[ri]);
            if (lane == 0) {
                m_s[r] = m_row[ri];
                l_s[r] = l;
            }
        }
    }
    __syncthreads();

    const bool single = p.num_splits == 1;
    for (int i = tid; i < p.R * D; i += kDecThreads) {
        const int r = i / D, d = i - (i / D) * D;
        float x = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) x += red[(w * RMAX + r) * D + d];
        const float l = l_s[r];
        const float o = l > 0.f ? x / l : 0.f;  // a row with no allowed key: O = 0
        if (single)
            p.o[row0 * D + i] = o;
        else
            p.o_part[(long long)blockIdx.x * p.R * D + i] = o;
    }
    if (tid < p.R) {
        const float l = l_s[tid];
        const float lse2 = l > 0.f ? m_s[tid] + log2f(l) : -INFINITY;
        if (single)
            p.lse[row0 + tid] = lse2 * 0.6931471805599453f;
        else
            p.l_part[(long long)blockIdx.x * p.R + tid] = lse2;
    }
}

// ------------------------------------------------------------------ merge kernel

// One warp per query row: O = sum_s w_s O_s / sum_s w_s with
// w_s = 2^(L_s - max_s L_s), and LSE = max_s L_s + log2(sum_s w_s), returned
// in natural-log units.  Partitions whose rows saw no allowed key carry
// L_s = -inf and weigh nothing; a row empty in every partition gets O = 0 and
// LSE = -inf (FlashAttention from Scratch, sec. 4.3, the empty case of the
// merge, and sec. 4.4).
template <int D>
__global__ void __launch_bounds__(256) fa_decode_merge_kernel(const DecodeParams p)
{
    constexpr int V = D / 32;  // dimensions per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 8 + warp;
    if (row >= (long long)p.B * p.Hkv * p.R) return;
    const int bh = (int)(row / p.R), r = (int)(row - (long long)bh * p.R);
    const int S = p.num_splits;
    const float* lp = p.l_part + (long long)bh * S * p.R + r;
    float mx = -INFINITY;
    for (int s = lane; s < S; s += 32) mx = fmaxf(mx, lp[(long long)s * p.R]);
    mx = warp_max(mx);
    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    if (mx != -INFINITY) {
        const float* op = p.o_part + ((long long)bh * S * p.R + r) * D + lane * V;
        for (int s0 = 0; s0 < S; s0 += 8) {
            // eight partitions' loads in flight before any is used
            float lv[8], x[8][V];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int s = min(s0 + u, S - 1);
                lv[u] = lp[(long long)s * p.R];
                const float* src = op + (long long)s * p.R * D;
                if constexpr (V == 4) {
                    const float4 t = *reinterpret_cast<const float4*>(src);
                    x[u][0] = t.x;
                    x[u][1] = t.y;
                    x[u][2] = t.z;
                    x[u][3] = t.w;
                } else {
                    const float2 t = *reinterpret_cast<const float2*>(src);
                    x[u][0] = t.x;
                    x[u][1] = t.y;
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (s0 + u < S) {  // partitions in order, as before the batching
                    const float w = ex2_approx(lv[u] - mx);
#pragma unroll
                    for (int e = 0; e < V; ++e) acc[e] = fmaf(w, x[u][e], acc[e]);
                    wsum += w;
                }
            }
        }
    }
    const int b = bh / p.Hkv, hkv = bh - b * p.Hkv;
    const long long orow = ((long long)b * p.Hq + (long long)hkv * p.group) * p.Lq + r;
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    float* dst = p.o + orow * D + lane * V;
    if constexpr (V == 4) {
        *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    } else {
        *reinterpret_cast<float2*>(dst) = make_float2(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0) p.lse[orow] = wsum > 0.f ? (mx + log2f(wsum)) * 0.6931471805599453f : -INFINITY;
}

// ------------------------------------------------------------------ host side

int decode_rows_per_thread(int D, int R)
{
    const int rg = 256 / D;
    for (int rpt = 1; rpt <= 8; rpt *= 2)
        if (rg * rpt >= R && rg * rpt <= kDecMaxRows) return rpt;
    return 0;
}

namespace {

template <int D, int RPT>
struct DecKernel {
    static constexpr int SMEM = DecSmem<D, DecCfg<D>::RG * RPT>::DYNAMIC;
    static cudaError_t prepare()
    {
        static_assert(SMEM <= 232448, "shared memory of one CTA");
        return smem_limit_once<fa_decode_partial_kernel<D, RPT>>(SMEM);
    }
    static cudaError_t launch(const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p, int grid,
                              cudaStream_t st)
    {
        const cudaError_t e = prepare();
        if (e != cudaSuccess) return e;
        fa_decode_partial_kernel<D, RPT><<<grid, kDecThreads, SMEM, st>>>(k, v, p);
        return cudaGetLastError();
    }
    static int occupancy()
    {
        if (prepare() != cudaSuccess) return 1;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fa_decode_partial_kernel<D, RPT>, kDecThreads, SMEM) !=
            cudaSuccess)
            return 1;
        return n > 0 ? n : 1;
    }
};

template <int D, typename F>
auto with_rpt(int rpt, F&& f)
{
    switch (rpt) {
        case 1: return f(DecKernel<D, 1>{});
        case 2: return f(DecKernel<D, 2>{});
        case 4: return f(DecKernel<D, 4>{});
        default: return f(DecKernel<D, (D == 128 ? 8 : 4)>{});
    }
}

constexpr int kMaxDev = 64;
std::mutex g_occ_mu;
int g_occ[kMaxDev][2][4];  // [device][D == 128][log2 rpt], 0 = not yet known

}  // namespace

int decode_ctas_per_sm(int D, int rpt)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 1;
    const int di = D == 128 ? 1 : 0;
    const int ri = rpt >= 8 ? 3 : rpt >= 4 ? 2 : rpt >= 2 ? 1 : 0;
    std::lock_guard<std::mutex> lock(g_occ_mu);
    int& slot = g_occ[dev][di][ri];
    if (slot == 0)
        slot = D == 128 ? with_rpt<128>(rpt, [](auto k) { return decltype(k)::occupancy(); })
                        : with_rpt<64>(rpt, [](auto k) { return decltype(k)::occupancy(); });
    return slot;
}

cudaError_t launch_decode_partial(int D, int rpt, const CUtensorMap& k, const CUtensorMap& v, const DecodeParams& p,
                                  int grid, cudaStream_t stream)
{
    if (D == 128)
        return with_rpt<128>(rpt, [&](auto kk) { return decltype(kk)::launch(k, v, p, grid, stream); });
    return with_rpt<64>(rpt, [&](auto kk) { return decltype(kk)::launch(k, v, p, grid, stream); });
}

cudaError_t launch_decode_merge(int D, const DecodeParams& p, cudaStream_t stream)
{
    const long long rows = (long long)p.B * p.Hkv * p.R;
    const int grid = (int)((rows + 7) / 8);
    if (D == 128)
        fa_decode_merge_kernel<128><<<grid, 256, 0, stream>>>(p);
    else
        fa_decode_merge_kernel<64><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace fa
