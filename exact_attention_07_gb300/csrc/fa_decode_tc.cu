// Split-KV decode partials on the fifth-generation tensor cores (sm_103a, D = 64 and 128).
//
// Grouped-query decode has R = (Hq / Hkv) * Lq query rows per KV head (up to
// 16 here).  Packing those rows into one work tile fills a matrix
// instruction's otherwise mostly empty query dimension (FlashAttention from
// Scratch, sec. 9.2 "GQA changes the reuse opportunity").  Keys take the
// 128-row side of the MMA and the packed query rows the 16-column side:
//
//     S^T [128 keys x 16 rows] = K_tile [128 x D] . Q^T [D x 16]
//     O^T [D x 16 rows]       += V_tile^T [D x 128] . P^T [128 keys x 16]
//
// both accumulating in tensor memory.  With D = 64 a tile holds 256 keys (two
// 128-key halves, each an S^T MMA of its own), so that a tile carries the same
// 64 KB of K and V as at D = 128 for about the same fixed softmax work per
// tile.  The second product then takes both halves in one MMA of M = 128,
// N = 32: A stacks V^T of the first half (dimensions on rows 0..63) over V^T
// of the second (rows 64..127), B puts P^T of the first half in columns 0..15
// and of the second in 16..31, and O^T is the sum of the two diagonal 64 x 16
// quadrants of the accumulator (the other two are cross terms, never read).
// A tile then takes 8 + 8 MMAs at either head dimension: each tcgen05.mma of
// these small shapes costs the issuing warp about 100 cycles here, which is
// what bounded a 256-key tile with 16 separate 16-key products.
// The tensor core does the contraction
// at a small fraction of its rate, so the kernel is bound by streaming K and
// V from HBM; the FP32-pipe variant (fa_decode.cu) runs out of issue slots
// first once R reaches 4.
//
// Roles (one persistent CTA per SM, work items = (batch, KV head, key
// partition) in a strided order), with G = 1 softmax warpgroup for up to 4
// carried rows and G = 2 (each carrying half of the rows) for 8 or 16:
//   warps 0..4G-1  softmax: in each group, thread k owns TMEM lane k -- key
//              k of each 128-key half for S^T, output dimension k for O^T
//              (D = 64: threads 64..127 hold the second half's partial sums
//              of dimension k - 64, added in the epilogue).  Row maxima
//              across the keys go through a transposing warp reduction and a
//              four-warp exchange in shared memory; P^T is written to shared
//              memory in the operand layout; O^T is rescaled in place when a
//              row's reference moves; the epilogue normalises and stores.
//              Only the first NR >= R of the 16 MMA columns are carried.
//   warp  4G    TMA producer: Q rows of the item, then K and V tiles in a ring.
//   warp  4G+1  S^T MMA issuer and tensor-memory owner.
//   warp  4G+2  O^T MMA issuer.
// The online-softmax state follows the dense kernel: base-2 exponentials,
// a per-row reference r that moves only when a tile maximum exceeds it by
// more than 8, the bf16-rounded probability sum to normalise O and the fp32
// sum for the log-sum-exp (FlashAttention from Scratch, sec. 4.2 and sec. 11.3).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fa_decode.h"
#include "ptx_sm103.cuh"

namespace fa {

namespace {

constexpr int kTcRows = 16;            // packed query rows (the MMA's N)
// Softmax warpgroups: one for up to 4 carried rows, two (rows split in
// halves) for 8 or 16, so that a thread's per-tile work stays small.  The
// producer and the two MMA warps follow them.
constexpr int tc_groups(int NR) { return NR > 4 ? 2 : 1; }
constexpr int tc_threads(int NR) { return 32 * (4 * tc_groups(NR) + 3); }
constexpr int kHalfBytes = 128 * 64 * 2;         // one [128 keys][64 dimensions] box: 16 KB
constexpr int kQBox = kTcRows * 64 * 2;          // one 64-dimension box of Q: 2 KB

// D = head dimension (64 or 128).  A tile is kKeys = 16384 / D keys (32 KB of
// K or of V), in kSub halves of 128 keys (the S^T MMA's M); the ring holds six
// tiles.  P^T is stored as 64-key swizzle atoms of kSub * 16 rows (row
// 16 u + r: query row r of half u), so that the O^T MMA reads both halves'
// probabilities as one operand of N = kSub * 16 columns.
template <int D>
struct TcSmem {
    static constexpr int kKeys = 16384 / D;                // keys per tile
    static constexpr int kSub = kKeys / 128;               // 128-key halves of a tile
    static constexpr int kBoxes = D / 64;                  // 64-dimension boxes per key row
    static constexpr int kSlotBytes = kKeys * D * 2;       // one K or V tile: 32 KB
    static constexpr int kNumSlots = 6;                    // K/V ring slots
    static constexpr int kQBytes = kTcRows * D * 2;
    static constexpr int kPAtom = kSub * kTcRows * 128;    // P^T: one 64-key atom of kSub * 16 rows
    static constexpr int kPBytes = 2 * kPAtom;             // P^T of one tile: two atoms
    static constexpr int kSlots = 0;
    static constexpr int kQ = kSlots + kNumSlots * kSlotBytes;       // [2] Q buffers
    static constexpr int kP = kQ + 2 * kQBytes;                      // [2] P^T buffers
    static constexpr int kRed = kP + 2 * kPBytes;              // float [2 buffers][2 groups][4][16] row maxima
    static constexpr int kEpi = kRed + 2 * 2 * 4 * 16 * 4;     // float [2 groups][4][32] row sums
    static constexpr int kSum = kEpi + 2 * 4 * 32 * 4;         // D = 64: float [16][64] second-half O^T
    static constexpr int kBars = kSum + (kSub == 2 ? kTcRows * 64 * 4 : 0);
    // barrier slots
    static constexpr int bQFull = 0, bQEmpty = 2, bKVFull = 4, bKVEmpty = 4 + kNumSlots;
    static constexpr int bSFull = 4 + 2 * kNumSlots, bSEmpty = bSFull + 2, bPFull = bSFull + 4,
                         bPEmpty = bSFull + 6, bOFull = bSFull + 8, bOEmpty = bSFull + 9,
                         bRed = bSFull + 10, bEpi = bSFull + 14, bDrain = bSFull + 16, kNumBars = bSFull + 18;
    // bRed + 2 * buffer + group, bEpi + group
    static constexpr int kMisc = kBars + kNumBars * 8;  // tmem base, abort flag
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kDynamic = kBytes + 1024;
    static_assert(kDynamic <= 232448, "shared memory of one CTA");
};

// TMEM columns: S^T double buffer (kSub groups of 16 columns each), then O^T
// (kSub groups of 16: at D = 64 lanes 0..63 of the first and lanes 64..127 of
// the second hold the two halves' partial sums).
template <int D>
struct TcTmem {
    static constexpr uint32_t kColS = 0, kColO = 2 * TcSmem<D>::kSub * kTcRows;
    static constexpr uint32_t kCols = kColO + TcSmem<D>::kSub * kTcRows <= 64 ? 64 : 128;  // a power of two >= 32
};

// tcgen05.ld / st of N = 4, 8 or 16 consecutive columns of this warp's 32 lanes.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N])
{
    uint32_t r[N];
    if constexpr (N == 4) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(taddr)
                     : "memory");
    } else if constexpr (N == 8) {
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                       "=r"(r[7])
                     : "r"(taddr)
                     : "memory");
    } else {
        static_assert(N == 16, "4, 8 or 16 columns");
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
            "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr)
            : "memory");
    }
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
}

template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const float (&v)[N])
{
    uint32_t r[N];
#pragma unroll
    for (int i = 0; i < N; ++i) r[i] = __float_as_uint(v[i]);
    if constexpr (N == 4) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]),
                     "r"(r[1]), "r"(r[2]), "r"(r[3])
                     : "memory");
    } else if constexpr (N == 8) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                     "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                     : "memory");
    } else {
        static_assert(N == 16, "4, 8 or 16 columns");
        asm volatile(
            "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
            "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
            "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
            "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
            : "memory");
    }
}

// Generic-proxy shared-memory writes become visible to the tensor core's
// (async proxy) operand reads.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v)
{
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ bool tc_warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             const WaitFailure& wf, int site, int item)
{
    const bool ok = mbar_wait(bar, parity, abort_flag, wf, site, item);
    return __all_sync(0xffffffffu, ok);
}

// Reduces N per-lane values (one per query row, N = 4, 8 or 16) across the
// warp with a transposing butterfly: each exchange halves the rows a lane
// carries, so N + N/2 + ... values cross lanes instead of N * 5.  Returns, in
// every lane, the reduction of row lane / (32 / N) over all 32 lanes.
template <bool MAX, int N>
__device__ __forceinline__ float transpose_reduce(const float (&v)[N], int lane)
{
    auto op = [](float a, float b) { return MAX ? fmaxf(a, b) : a + b; };
    float c[N];
#pragma unroll
    for (int i = 0; i < N; ++i) c[i] = v[i];
    int mask = 16;
#pragma unroll
    for (int w = N; w > 1; w >>= 1, mask >>= 1) {
        const bool upper = lane & mask;  // this lane keeps the upper half of the rows it carries
#pragma unroll
        for (int i = 0; i < w / 2; ++i) {
            const float send = upper ? c[i] : c[i + w / 2], keep = upper ? c[i + w / 2] : c[i];
            c[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, mask));
        }
    }
    float d = c[0];
#pragma unroll
    for (; mask >= 1; mask >>= 1) d = op(d, __shfl_xor_sync(0xffffffffu, d, mask));
    return d;
}

struct TcItem {
    int bh, split, t0, n;
    long long row0;
};

__device__ __forceinline__ TcItem tc_item(const DecodeParams& p, int it)
{
    TcItem w;
    w.bh = it / p.num_splits;
    w.split = it - w.bh * p.num_splits;
    w.t0 = w.split * p.tiles_per_split;
    w.n = min(p.num_tiles - w.t0, p.tiles_per_split);
    const int b = w.bh / p.Hkv, hkv = w.bh - b * p.Hkv;
    w.row0 = ((long long)b * p.Hq + (long long)hkv * p.group) * p.Lq;
    return w;
}

}  // namespace

// NR = query rows the softmax carries (4, 8 or 16 >= R); the MMAs keep N = 16,
// and the rows of P^T past NR stay zero.
template <int D, int NR>
__global__ void __launch_bounds__(tc_threads(NR), 1)
    fa_decode_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecodeParams p)
{
    using L = TcSmem<D>;
    constexpr int kTcSlots = L::kNumSlots, kSlotBytes = L::kSlotBytes, kQBytes = L::kQBytes;
    constexpr int kKeys = L::kKeys, kSub = L::kSub, kPBytes = L::kPBytes, kPAtom = L::kPAtom;
    constexpr uint32_t kColS = TcTmem<D>::kColS, kColO = TcTmem<D>::kColO, kTmemCols = TcTmem<D>::kCols;
    constexpr float kTau = 8.0f;
    constexpr int NG = tc_groups(NR), RG = NR / NG;  // softmax groups, rows of each
    constexpr int kLanesPerRow = 32 / RG;  // lanes that end a transposing reduction with the same row
    constexpr int kThreads = tc_threads(NR);
    constexpr int wProd = 4 * NG, wMmaS = 4 * NG + 1, wMmaPV = 4 * NG + 2;  // warp roles after the softmax
    static_assert(wMmaPV == kThreads / 32 - 1, "the O^T MMA warp is the last");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sb + L::kBars + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
    float* red = reinterpret_cast<float*>(smem + L::kRed);
    float* epi = reinterpret_cast<float*>(smem + L::kEpi);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WaitFailure wf{p.err, p.diag};
    const int num_items = p.B * p.Hkv * p.num_splits;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(L::bQFull + i), 1);
            mbar_init(bar(L::bQEmpty + i), 1);
            mbar_init(bar(L::bSFull + i), 1);
            mbar_init(bar(L::bSEmpty + i), 128 * NG);
            mbar_init(bar(L::bPFull + i), 128 * NG);
            mbar_init(bar(L::bPEmpty + i), 1);
            mbar_init(bar(L::bRed + 2 * i), 128);
            mbar_init(bar(L::bRed + 2 * i + 1), 128);
            mbar_init(bar(L::bEpi + i), 128);
        }
        for (int s = 0; s < kTcSlots; ++s) {
            mbar_init(bar(L::bKVFull + s), 1);
            mbar_init(bar(L::bKVEmpty + s), 1);
        }
        mbar_init(bar(L::bOFull), 1);
        mbar_init(bar(L::bOEmpty), 128 * NG);
        mbar_init(bar(L::bDrain), 1);
        mbar_init(bar(L::bDrain + 1), 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == wProd && lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
    }
    if (warp == wMmaS) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if constexpr (NR < kTcRows) {
        // P^T rows NR..15 are never written: zeros for the O^T MMA
        uint4* z = reinterpret_cast<uint4*>(smem + L::kP);
        for (int i = threadIdx.x; i < 2 * kPBytes / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp < 4 * NG) {
        // ============================================================ softmax
        // group g carries query rows g*RG .. g*RG + RG - 1 of the 16
        const int g = warp >> 2, wq = warp & 3;
        const int k = 32 * wq + lane;  // TMEM lane: key of the tile / output dimension
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        // this thread's O^T columns: D = 64 lanes 64..127 hold the second half's partial sums
        const uint32_t col_o = kColO + (kSub == 2 && wq >= 2 ? (uint32_t)kTcRows : 0u) + (uint32_t)(g * RG);
        const int row0 = g * RG;  // first query row of the group
        const int causal_off = p.Lk - p.Lq;
        // last key each row may see (bottom-right causal alignment, padding at Lk)
        int lim[RG];
        int lim_min = p.Lk - 1;
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            lim[r] = p.causal ? min(p.Lk - 1, ((row0 + r) % p.Lq) + causal_off) : p.Lk - 1;
            if (row0 + r < p.R) lim_min = min(lim_min, lim[r]);
        }
        uint32_t T = 0;
        int I = 0;
        for (int it = blockIdx.x; it < num_items; it += gridDim.x, ++I) {
            const TcItem w = tc_item(p, it);
            float ref[RG], lf[RG], lb[RG];
#pragma unroll
            for (int r = 0; r < RG; ++r) {
                ref[r] = -INFINITY;
                lf[r] = 0.f;
                lb[r] = 0.f;
            }
            for (int t = 0; t < w.n; ++t, ++T) {
                const uint32_t b = T & 1u, ph = (T >> 1) & 1u;
                if (!tc_warp_wait(bar(L::bSFull + b), ph, abort_flag, wf, 60, it)) goto done;
                tc_fence_after_sync();
                // this thread's keys: k + 128 u of the tile, u < kSub
                float s[kSub][RG];
#pragma unroll
                for (int u = 0; u < kSub; ++u)
                    tmem_ld_cols<RG>(lane_base + kColS + (b * kSub + u) * kTcRows + row0, s[u]);
                tmem_wait_ld();
                tc_fence_before_sync();
                mbar_arrive(bar(L::bSEmpty + b));
                const int key_base = (w.t0 + t) * kKeys;
#pragma unroll
                for (int u = 0; u < kSub; ++u)
#pragma unroll
                    for (int r = 0; r < RG; ++r) s[u][r] *= p.scale_log2;
                if (key_base + kKeys - 1 > lim_min) {  // tile reaches masked keys
#pragma unroll
                    for (int u = 0; u < kSub; ++u)
#pragma unroll
                        for (int r = 0; r < RG; ++r)
                            if (key_base + 128 * u + k > lim[r]) s[u][r] = -INFINITY;
                }
                // tile maximum of every row over the tile's keys
                float sm[RG];
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    sm[r] = s[0][r];
#pragma unroll
                    for (int u = 1; u < kSub; ++u) sm[r] = fmaxf(sm[r], s[u][r]);
                }
                const float wm = transpose_reduce<true>(sm, lane);
                float* rb = red + (2 * b + g) * 64;
                if (lane % kLanesPerRow == 0) rb[wq * 16 + lane / kLanesPerRow] = wm;
                mbar_arrive(bar(L::bRed + 2 * b + g));
                if (!tc_warp_wait(bar(L::bRed + 2 * b + g), ph, abort_flag, wf, 61, it)) goto done;
                float tm_lane = -INFINITY;
                if (lane < RG)
                    tm_lane = fmaxf(fmaxf(rb[lane], rb[16 + lane]), fmaxf(rb[32 + lane], rb[48 + lane]));
                float alpha[RG];
                bool moved = false;
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    const float tm = __shfl_sync(0xffffffffu, tm_lane, r);
                    alpha[r] = 1.f;
                    if (tm > ref[r] + kTau) {  // also when ref is still -inf and the tile has a key
                        alpha[r] = ex2_approx(ref[r] - tm);
                        ref[r] = tm;
                        moved = true;
                    }
                }
                // probabilities, rounded to bf16 for the MMA; both sums
                uint32_t pk[kSub][RG / 2];
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    lf[r] *= alpha[r];
                    lb[r] *= alpha[r];
                }
#pragma unroll
                for (int u = 0; u < kSub; ++u)
#pragma unroll
                    for (int r = 0; r < RG; r += 2) {
                        const float p0 = ref[r] == -INFINITY ? 0.f : ex2_approx(s[u][r] - ref[r]);
                        const float p1 = ref[r + 1] == -INFINITY ? 0.f : ex2_approx(s[u][r + 1] - ref[r + 1]);
                        __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
                        pk[u][r / 2] = *reinterpret_cast<uint32_t*>(&h);
                        lf[r] += p0;
                        lf[r + 1] += p1;
                        lb[r] += __uint_as_float(pk[u][r / 2] << 16);
                        lb[r + 1] += __uint_as_float(pk[u][r / 2] & 0xffff0000u);
                    }
                // P^T buffer b is free once P.V of tile T - 2 has completed
                if (!tc_warp_wait(bar(L::bPEmpty + b), ph ^ 1u, abort_flag, wf, 62, it)) goto done;
                {
                    // key k of each half: atom k / 64, operand row 16 u + r
                    const uint32_t pb = sb + L::kP + b * kPBytes + (uint32_t)((k >> 6) * kPAtom) +
                                        (uint32_t)((k & 7) * 2);
                    const int chunk = (k & 63) >> 3;
#pragma unroll
                    for (int u = 0; u < kSub; ++u)
#pragma unroll
                        for (int r = 0; r < RG; ++r) {
                            const uint16_t h =
                                (r & 1) ? (uint16_t)(pk[u][r / 2] >> 16) : (uint16_t)(pk[u][r / 2] & 0xffffu);
                            const int n = 16 * u + row0 + r;  // operand row
                            sts16(pb + (uint32_t)(n * 128 + ((chunk ^ (n & 7)) << 4)), h);
                        }
                }
                fence_proxy_async_smem();
                if (moved && t > 0) {
                    // O^T holds tiles up to T - 1: wait for that P.V, then rescale in place
                    const uint32_t bp = (T - 1) & 1u, php = ((T - 1) >> 1) & 1u;
                    if (!tc_warp_wait(bar(L::bPEmpty + bp), php, abort_flag, wf, 63, it)) goto done;
                    tc_fence_after_sync();
                    float o[RG];
                    tmem_ld_cols<RG>(lane_base + col_o, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int r = 0; r < RG; ++r) o[r] *= alpha[r];
                    tmem_st_cols<RG>(lane_base + col_o, o);
                    tmem_wait_st();
                }
                tc_fence_before_sync();
                mbar_arrive(bar(L::bPFull + b));
            }
            // ---- epilogue of the item: O = O^T / l_rounded, LSE = r + log2(l)
            if (!tc_warp_wait(bar(L::bOFull), (uint32_t)(I & 1), abort_flag, wf, 64, it)) goto done;
            tc_fence_after_sync();
            float o[RG];
            tmem_ld_cols<RG>(lane_base + col_o, o);
            tmem_wait_ld();
            tc_fence_before_sync();
            mbar_arrive(bar(L::bOEmpty));
            float* osum = reinterpret_cast<float*>(smem + L::kSum);
            if (kSub == 2 && k >= 64) {
#pragma unroll
                for (int r = 0; r < RG; ++r) osum[(row0 + r) * 64 + (k - 64)] = o[r];
            }
            {
                const float sb_w = transpose_reduce<false>(lb, lane);
                const float sf_w = transpose_reduce<false>(lf, lane);
                if (lane % kLanesPerRow == 0) {
                    epi[g * 128 + wq * 32 + lane / kLanesPerRow] = sb_w;
                    epi[g * 128 + wq * 32 + 16 + lane / kLanesPerRow] = sf_w;
                }
            }
            mbar_arrive(bar(L::bEpi + g));
            if (!tc_warp_wait(bar(L::bEpi + g), (uint32_t)(I & 1), abort_flag, wf, 65, it)) goto done;
            // lane < 16: the rounded sums of the group's rows, else the fp32 sums
            const float* eg = epi + g * 128;
            const float lsum = eg[lane] + eg[32 + lane] + eg[64 + lane] + eg[96 + lane];
            if (kSub == 2 && k < 64) {
#pragma unroll
                for (int r = 0; r < RG; ++r) o[r] += osum[(row0 + r) * 64 + k];
            }
            const bool single = p.num_splits == 1;
#pragma unroll
            for (int r = 0; r < RG; ++r) {
                const float l_r = __shfl_sync(0xffffffffu, lsum, r);
                const float lf_r = __shfl_sync(0xffffffffu, lsum, 16 + r);
                const int rr = row0 + r;  // query row of the item
                if (rr < p.R) {
                    const float val = l_r > 0.f ? o[r] / l_r : 0.f;
                    if (k < D) {
                        if (single)
                            p.o[(w.row0 + rr) * D + k] = val;
                        else
                            p.o_part[((long long)it * p.R + rr) * D + k] = val;
                    }
                    if (k == r) {
                        const float lse2 = lf_r > 0.f ? ref[r] + log2f(lf_r) : -INFINITY;
                        if (single)
                            p.lse[w.row0 + rr] = lse2 * 0.6931471805599453f;
                        else
                            p.l_part[(long long)it * p.R + rr] = lse2;
                    }
                }
            }
        }
    } else if (warp == wProd) {
        // ============================================================ TMA producer
        if (lane == 0) {
            int q_armed[2] = {-1, -1};
            int kv_armed[kTcSlots];
            for (int s = 0; s < kTcSlots; ++s) kv_armed[s] = -1;
            int stage = 0;
            uint32_t kv_ph = 0;
            bool drop_first = p.fault == 1;  // test hook: the first K tile never arrives
            int I = 0;
            auto load = [&](const CUtensorMap* map, int key0, int bh, int it) -> bool {
                if (!mbar_wait(bar(L::bKVEmpty + stage), kv_ph ^ 1u, abort_flag, wf, 66, it)) return false;
                if (drop_first) {
                    drop_first = false;
                } else {
                    mbar_arrive_expect_tx(bar(L::bKVFull + stage), kSlotBytes);
                    kv_armed[stage] = (int)kv_ph;
                    const uint32_t dst = sb + L::kSlots + (uint32_t)(stage * kSlotBytes);
                    // two [128 keys][64 dimensions] boxes: the dimension halves
                    // (D = 128) or the key halves (D = 64, 256 keys)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        tma_load_3d(dst + h * kHalfBytes, map, bar(L::bKVFull + stage), L::kSub == 1 ? 64 * h : 0,
                                    L::kSub == 1 ? key0 : key0 + 128 * h, bh);
                }
                if (++stage == kTcSlots) {
                    stage = 0;
                    kv_ph ^= 1u;
                }
                return true;
            };
            for (int it = blockIdx.x; it < num_items; it += gridDim.x, ++I) {
                const TcItem w = tc_item(p, it);
                const int qb = I & 1;
                const uint32_t qph = (uint32_t)((I >> 1) & 1);
                if (!mbar_wait(bar(L::bQEmpty + qb), qph ^ 1u, abort_flag, wf, 67, it)) break;
                mbar_arrive_expect_tx(bar(L::bQFull + qb), kQBytes);
                q_armed[qb] = (int)qph;
                const uint32_t qdst = sb + L::kQ + (uint32_t)(qb * kQBytes);
#pragma unroll
                for (int h = 0; h < L::kBoxes; ++h)
                    tma_load_3d(qdst + h * kQBox, &tmQ, bar(L::bQFull + qb), 64 * h, (int)w.row0, 0);
                bool ok = true;
                for (int t = 0; t < w.n && ok; ++t) {
                    const int key0 = (w.t0 + t) * kKeys;
                    ok = load(&tmK, key0, w.bh, it) && load(&tmV, key0, w.bh, it);
                }
                if (!ok) break;
            }
            // every copy this thread started has landed before the CTA retires
            for (int i = 0; i < 2; ++i)
                if (q_armed[i] >= 0) mbar_settle(bar(L::bQFull + i), (uint32_t)q_armed[i], wf, 68);
            for (int s = 0; s < kTcSlots; ++s)
                if (kv_armed[s] >= 0) mbar_settle(bar(L::bKVFull + s), (uint32_t)kv_armed[s], wf, 69);
        }
        __syncwarp();
    } else {
        // ============================================================ MMA issuers
        // Warp 5 issues S^T, warp 6 the O^T update: each tcgen05.mma of these
        // shapes takes about as long to issue as to run, and a tile needs
        // 8 + 16 of them at D = 64.  K(T) and V(T) are loads 2T and 2T + 1 of
        // the ring.
        const bool leader = lane == 0;
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        const bool s_warp = warp == wMmaS;
        auto ring = [&](uint32_t n, int& slot, uint32_t& ph) {
            slot = (int)(n % (uint32_t)kTcSlots);
            ph = (n / (uint32_t)kTcSlots) & 1u;
        };
        auto commit = [&](int b) {
            if (leader) tc_commit(bar(b));
            __syncwarp();
        };
        uint32_t T = 0;
        bool issued = false, ok = true;
        int I = 0;
        for (int it = blockIdx.x; it < num_items && ok; it += gridDim.x, ++I) {
            const TcItem w = tc_item(p, it);
            const int qb = I & 1;
            if (s_warp) {
                constexpr uint32_t kIdescS = idesc_bf16_f32(128, kTcRows, false);
                if (!tc_warp_wait(bar(L::bQFull + qb), (uint32_t)((I >> 1) & 1), abort_flag, wf, 73, it)) break;
                const uint64_t qd = smem_desc_sw128(sb + L::kQ + (uint32_t)(qb * kQBytes), 16, 1024);
                for (int t = 0; t < w.n; ++t, ++T) {
                    int ks;
                    uint32_t kph;
                    ring(2 * T, ks, kph);
                    const uint32_t b = T & 1u;
                    if (!(ok = tc_warp_wait(bar(L::bKVFull + ks), kph, abort_flag, wf, 74, it))) break;
                    if (!(ok = tc_warp_wait(bar(L::bSEmpty + b), ((T >> 1) & 1u) ^ 1u, abort_flag, wf, 75, it)))
                        break;
                    tc_fence_after_sync();
                    const uint64_t kd = smem_desc_sw128(sb + L::kSlots + (uint32_t)(ks * kSlotBytes), 16, 1024);
                    if (leader) {
                        // S^T of each 128-key half: keys on the MMA's M, D/16 steps of K
#pragma unroll
                        for (int u = 0; u < kSub; ++u)
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint64_t koff =
                                    (uint64_t)((u * kHalfBytes + (kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
                                const uint64_t qoff = (uint64_t)(((kk >> 2) * kQBox + (kk & 3) * 32) >> 4);
                                mma_ss(tm + kColS + (b * kSub + u) * kTcRows, kd + koff, qd + qoff, kIdescS,
                                       kk > 0 ? 1u : 0u);
                            }
                    }
                    __syncwarp();
                    issued = true;
                    commit(L::bSFull + b);
                    commit(L::bKVEmpty + ks);
                    if (t == w.n - 1) commit(L::bQEmpty + qb);
                }
            } else {
                // A (V^T) MN-major; N = 32 at D = 64 (both key halves)
                constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kSub * kTcRows, false) | (1u << 15);
                for (int t = 0; t < w.n; ++t, ++T) {
                    int vs;
                    uint32_t vph;
                    ring(2 * T + 1, vs, vph);
                    const uint32_t bp = T & 1u;
                    if (!(ok = tc_warp_wait(bar(L::bKVFull + vs), vph, abort_flag, wf, 70, it))) break;
                    if (!(ok = tc_warp_wait(bar(L::bPFull + bp), (T >> 1) & 1u, abort_flag, wf, 71, it))) break;
                    if (t == 0 &&
                        !(ok = tc_warp_wait(bar(L::bOEmpty), (uint32_t)(I & 1) ^ 1u, abort_flag, wf, 72, it)))
                        break;
                    tc_fence_after_sync();
                    // A = V^T, MN-major, 16 keys (2 KB) per step; rows 64..127 are the
                    // second box, 16 KB on: dimensions 64..127 (D = 128) or keys
                    // 128..255 (D = 64)
                    const uint64_t vd =
                        smem_desc_sw128(sb + L::kSlots + (uint32_t)(vs * kSlotBytes), kHalfBytes, 1024);
                    const uint64_t pd = smem_desc_sw128(sb + L::kP + bp * kPBytes, 16, 1024);
                    if (leader) {
#pragma unroll
                        for (int kk = 0; kk < kKeys / (16 * kSub); ++kk) {
                            const uint64_t poff = (uint64_t)(((kk >> 2) * kPAtom + (kk & 3) * 32) >> 4);
                            mma_ss(tm + kColO, vd + (uint64_t)((kk * 16 * 128) >> 4), pd + poff, kIdescPV,
                                   (t == 0 && kk == 0) ? 0u : 1u);
                        }
                    }
                    __syncwarp();
                    issued = true;
                    commit(L::bPEmpty + bp);
                    commit(L::bKVEmpty + vs);
                }
                if (ok) commit(L::bOFull);
            }
        }
        // every MMA this warp issued has completed before TMEM is released
        if (issued) {
            const int db = L::bDrain + (s_warp ? 0 : 1);
            commit(db);
            mbar_settle(bar(db), 0, wf, 76);
        }
        __syncwarp();
    }
done:
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == wMmaS) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int NR>
cudaError_t launch_decode_tc_rows(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                  const DecodeParams& p, int grid, cudaStream_t stream)
{
    const cudaError_t e = smem_limit_once<fa_decode_tc_kernel<D, NR>>(TcSmem<D>::kDynamic);
    if (e != cudaSuccess) return e;
    fa_decode_tc_kernel<D, NR><<<grid, tc_threads(NR), TcSmem<D>::kDynamic, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_tc_dim(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const DecodeParams& p, int grid, cudaStream_t stream)
{
    if (p.R <= 4) return launch_decode_tc_rows<D, 4>(q, k, v, p, grid, stream);
    if (p.R <= 8) return launch_decode_tc_rows<D, 8>(q, k, v, p, grid, stream);
    return launch_decode_tc_rows<D, 16>(q, k, v, p, grid, stream);
}

cudaError_t launch_decode_tc(int D, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const DecodeParams& p, int grid, cudaStream_t stream)
{
    return D == 64 ? launch_decode_tc_dim<64>(q, k, v, p, grid, stream)
                   : launch_decode_tc_dim<128>(q, k, v, p, grid, stream);
}

}  // namespace fa
