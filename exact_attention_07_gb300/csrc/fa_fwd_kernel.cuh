// Exact attention forward for sm_103a (GB300): TMA -> shared-memory ring ->
// tcgen05 MMAs accumulating in tensor memory, online softmax one thread per
// query row, persistent CTAs over a longest-first tile order.
//
// Method (FlashAttention Cheat Sheet, sec. 4 "The complete FlashAttention
// flow" and sec. 5 "Why online softmax is globally exact"; FlashAttention
// from Scratch, sec. 6.3 "Build a small fused forward" and sec. 7.1 "Delay
// normalization"): a CTA keeps its query rows resident, streams K and V tiles
// past them, keeps per row a running reference r, a running sum l and an
// unnormalised accumulator A, and writes O = A / l and LSE = r + ln l once.
// Scores S and probabilities P live only in tensor memory.
//
// Work split inside a CTA (FlashAttention-4: Blackwell Attention Kernel Co-Design, "Forward TMEM pipeline"):
//   warps 0-3   softmax for Q tile 0 (rows 0..127 of the CTA's 256-row block)
//   warps 4-7   softmax for Q tile 1 (rows 128..255)
//   warps 8-11  epilogue: O = A / l -> fp32 -> global, LSE
//   warp  12    TMA producer: Q tiles and the K/V ring
//   warp  13    MMA issuer and tensor-memory owner
//   warps 14-15 idle
// Register budget per thread after setmaxnreg, the whole register file at the
// launch's 128 per thread: softmax 192, epilogue 64, producer/MMA warpgroup 64
// (2*128*192 + 128*64 + 128*64 = 65536); a few kernels shift it (kSmRegs,
// kEpiRegs, kCtlRegs in the kernel body).
// The two Q tiles ping-pong: while one softmax group turns S into P, the
// tensor core computes the other tile's S or P.V.
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [0,128)   S0 (fp32); P0 (bf16 pairs) overwrites its first 64 columns
//   [128,256) S1 / P1
//   [256,256+DV)       O0 accumulator (fp32), DV = value head dimension
//   [256+DV,256+2DV)   O1 accumulator
//
// Base-2 exponentials with log2(e) folded into the scale (FlashAttention from
// Scratch, sec. 6.3): p = 2^(s * scale * log2e - r).  The reference r only
// moves when a tile's maximum exceeds it by more than 8 (a factor 256;
// sec. 11.3 "Derive conditional rescaling correctly"), so O rarely needs a
// correction; when it does, the softmax thread that owns the row rescales it
// in tensor memory before releasing P.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_params.h"
#include "ptx_sm103.cuh"

namespace fa {

// Shared-memory layout.  D = query/key head dimension, DV = value head
// dimension (DV < D in the (192, 128) case).  The K/V ring holds V tiles and
// the first DV columns of K tiles; when D > DV the remaining K columns go
// through a second, smaller ring.
template <int D, int VAR = kVarNone, int DV = D>
struct FwdSmem {
    static constexpr bool kFp8 = VAR == kVarFp8;
    static constexpr int kElem = kFp8 ? 1 : 2;                      // bytes per element
    static constexpr int kBlk = kBlockN * 128;                      // 128 rows of one 128-byte swizzle block
    static constexpr int kQBytes = kBlockM * D * kElem;             // one Q tile
    static constexpr int kTileBytes = kBlockN * DV * kElem;         // one ring stage
    static constexpr int kTailBytes = kBlockN * (D - DV) * kElem;   // one stage of the K-tail ring
    static constexpr bool kTail = kTailBytes > 0;
    static constexpr int kHalvesQ = kQBytes / kBlk;                 // swizzle blocks per Q row
    static constexpr int kHalves = kTileBytes / kBlk;               // swizzle blocks per ring-stage row
    static constexpr int kTailHalves = kTailBytes / kBlk;
    static constexpr int kStages = kTail ? 3 : (kTileBytes == 32768 ? 4 : 8);  // K/V ring depth
    static constexpr int kTailStages = kTail ? 2 : 0;
    static constexpr int kQOff = 0;                                 // Q0, Q1
    static constexpr int kKVOff = 2 * kQBytes;
    static constexpr int kTailOff = kKVOff + kStages * kTileBytes;
    static constexpr int kPOff = kTailOff + kTailStages * kTailBytes;  // FP8: P0, P1 (e4m3, A of P.V)
    static constexpr int kBarOff = kPOff + (kFp8 ? 2 * kTileBytes : 0);
    // barrier slots (8 bytes each)
    static constexpr int kQFull = 0, kQEmpty = 2, kKVFull = 4, kKVEmpty = 4 + kStages;
    static constexpr int kTFull = 4 + 2 * kStages, kTEmpty = kTFull + kTailStages;
    static constexpr int kSFull = kTFull + 2 * kTailStages, kPFull = kSFull + 2, kOFull = kSFull + 4,
                         kOEmpty = kSFull + 6, kStFull = kSFull + 8, kStEmpty = kSFull + 10,
                         kDrain = kSFull + 12, kSEmpty = kSFull + 13, kPEmpty = kSFull + 15,
                         kNumBars = kSFull + 17;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;      // tmem base, abort flag
    static constexpr int kStatsOff = (kMiscOff + 16 + 15) / 16 * 16;  // float2 [2][128]
    // epilogue staging: per epilogue warp one 32 x 32 fp32 block, rows padded
    // to 36 floats (conflict-free 16-byte accesses by row and by column group);
    // left out where shared memory has no room for it (D > DV) and for e4m3
    // inputs (the epilogue's 64 registers then spill; measured slower)
    static constexpr int kEpiRowBytes = 36 * 4, kEpiWarpBytes = 32 * kEpiRowBytes;
    static constexpr bool kEpiStaged = !kTail && !kFp8;
    static constexpr int kEpiOff = kStatsOff + 2 * kBlockM * 8;
    static constexpr int kBytes = kEpiOff + (kEpiStaged ? 4 * kEpiWarpBytes : 0);
    // 1 KB of slack for aligning the window where it fits; otherwise the kernel
    // checks the alignment at run time
    static constexpr int kMaxDynamic = 232448;
    static constexpr int kAlloc = kBytes + 1024 <= kMaxDynamic ? kBytes + 1024 : kMaxDynamic;
    static_assert(kBytes <= kMaxDynamic, "shared-memory layout exceeds the per-CTA limit");
    static constexpr uint32_t kTmemCols = 512;
    // P in tensor-memory columns of its own (head dimension 64, bf16 inputs):
    // S_t [128 t, 128 t + 128), P_t [256 + 64 t, ...), O_t [384 + 64 t, ...).
    // The MMA warp can then compute S_t(j+1) as soon as the softmax has read
    // S_t(j), while that softmax is still turning it into P_t(j).  Elsewhere P_t
    // overwrites the first half of S_t and O_t sits at 256 + DV t.
    static constexpr bool kSplitP = D == 64 && DV == 64 && !kFp8;
    static constexpr uint32_t kColS = 0, kColP = kSplitP ? 256 : 0, kColO = kSplitP ? 384 : 256;
    static constexpr uint32_t kPStride = kSplitP ? 64 : kBlockN;  // columns between P_0 and P_1
    static_assert(kColO + 2 * DV <= kTmemCols, "tensor-memory layout");
};

// Schedule of a packed batch built by the CTA itself (launches without a
// precomputed schedule): tile prefix by rank [n + 1] and rank -> sequence
// [n], placed after every other region of the layout.  While it is being
// built, the K/V ring (not yet loaded) serves as scratch for the sort.
template <int D, int VAR, int DV>
struct FwdSchedSmem {
    using L = FwdSmem<D, VAR, DV>;
    static constexpr int kMaxSeqs = varlen_sched_max_seqs(D, DV);
    static constexpr int kOff = (L::kBytes + 15) / 16 * 16;
    static constexpr int kBytes = kOff + (2 * kMaxSeqs + 1) * 4;
    static constexpr int kAlloc = kBytes + 1024 <= L::kMaxDynamic ? kBytes + 1024 : L::kMaxDynamic;
    static_assert(kBytes <= L::kMaxDynamic, "packed-batch schedule exceeds the per-CTA shared memory");
    // sort scratch in the ring: 64-bit keys of the padded count, tiles per sequence, 32 warp sums
    static constexpr int kPad = kMaxSeqs <= 64 ? 64 : (kMaxSeqs <= 2048 ? 2048 : 4096);
    static_assert(kPad >= kMaxSeqs, "sort padding");
    static_assert(kPad * 12 + 32 * 4 <= L::kStages * L::kTileBytes, "sort scratch exceeds the ring");
};

// Dynamic shared memory of one forward kernel instance.
template <int D, bool VARLEN, int VAR, int DV>
constexpr int fwd_smem_alloc()
{
    return VARLEN ? FwdSchedSmem<D, VAR, DV>::kAlloc : FwdSmem<D, VAR, DV>::kAlloc;
}

__device__ __forceinline__ int ld_shared_s32(uint32_t addr)
{
    int v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// The packed batch's schedule: the precomputed one in global memory
// (p.sched), else the one this CTA built at shared address `ss` (tile prefix
// by rank [n + 1], then rank -> sequence [n]).  Read through the kernel
// parameters and a 32-bit shared address, so no pointer stays live in the
// roles' registers.
struct VarSchedView {
    const FwdParams& p;
    uint32_t ss;
    __device__ __forceinline__ bool pre() const { return p.sched != nullptr; }
    __device__ __forceinline__ int n() const { return pre() ? p.num_seqs : p.seq_count; }
    __device__ __forceinline__ int prefix(int r) const
    {
        return pre() ? __ldg(p.sched + 1 + r) : ld_shared_s32(ss + 4u * (uint32_t)r);
    }
    __device__ __forceinline__ int order(int r) const
    {
        return pre() ? __ldg(p.sched + 2 + p.num_seqs + r) : ld_shared_s32(ss + 4u * (uint32_t)(p.seq_count + 1 + r));
    }
};

// Builds the schedule of sequences [p.seq_begin, p.seq_begin + p.seq_count)
// with every thread of the CTA: validates their offsets, orders them by key
// length, longest first (FlashAttention-4: Blackwell Attention Kernel
// Co-Design, "LPT scheduling for imbalanced grids"; ties keep the batch
// order), and writes the exclusive prefix of work tiles (Hq * ceil(Lq / 256)
// per sequence) in that order.  An invalid sequence, or any sequence when the
// offsets do not start at 0 and end at the totals, is given no work and sets
// error bit 1.  `keys` holds kPad 64-bit entries, `tiles` kPad + 32 ints.
template <int kPad>
__device__ __forceinline__ void build_varlen_schedule(const FwdParams& p, unsigned long long* keys, int* tiles,
                                                      int* prefix, int* order)
{
    const int n = p.seq_count, tid = (int)threadIdx.x, nthr = (int)blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
    int npad = 2;
    while (npad < n) npad <<= 1;
    const bool bad = __ldg(p.cu_q) != 0 || __ldg(p.cu_k) != 0 || __ldg(p.cu_q + p.num_seqs) != p.total_q ||
                     __ldg(p.cu_k + p.num_seqs) != p.total_k;
    for (int i = tid; i < npad; i += nthr) {
        unsigned long long key = ~0ull;
        if (i < n) {
            const int s = p.seq_begin + i;
            const int q0 = __ldg(p.cu_q + s), q1 = __ldg(p.cu_q + s + 1);
            const int k0 = __ldg(p.cu_k + s), k1 = __ldg(p.cu_k + s + 1);
            const bool ok = !bad && q0 >= 0 && q1 >= q0 && q1 <= p.total_q && q1 - q0 <= p.max_q && k0 >= 0 &&
                            k1 >= k0 && k1 <= p.total_k && k1 - k0 <= p.max_k;
            if (!ok && blockIdx.x == 0) atomicOr(p.err, 2);
            const int len = (ok && q1 > q0) ? (k1 - k0) : -1;
            tiles[i] = !ok ? 0
                       : p.pair_heads ? (p.Hq >> 1) * ((q1 - q0 + kBlockM - 1) / kBlockM)
                                      : p.Hq * ((q1 - q0 + kRowsPerCta - 1) / kRowsPerCta);
            // ascending order of (longest first, then batch order)
            key = ((unsigned long long)(0x7fffffffu - (unsigned)len) << 32) | (unsigned)i;
        }
        keys[i] = key;
    }
    __syncthreads();
    // bitonic sort of keys[0 .. npad)
    for (int k = 2; k <= npad; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < npad; i += nthr) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long a = keys[i], b = keys[ixj];
                    if ((a > b) == ((i & k) == 0)) {
                        keys[i] = b;
                        keys[ixj] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    // rank -> sequence, and an exclusive scan of the tiles in rank order:
    // each thread takes a run of consecutive ranks
    const int per = (n + nthr - 1) / nthr;
    const int r0 = min(n, tid * per), r1 = min(n, r0 + per);
    int sum = 0;
    for (int r = r0; r < r1; ++r) {
        const int i = (int)(unsigned)keys[r];
        order[r] = p.seq_begin + i;
        sum += tiles[i];
    }
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    int* wsum = tiles + kPad;
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int x = lane < nwarps ? wsum[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, d);
            if (lane >= d) x += y;
        }
        wsum[lane] = x;
    }
    __syncthreads();
    int acc = (warp > 0 ? wsum[warp - 1] : 0) + incl - sum;
    for (int r = r0; r < r1; ++r) {
        prefix[r] = acc;
        acc += tiles[(int)(unsigned)keys[r]];
    }
    if (tid == 0) prefix[n] = wsum[nwarps - 1];
}

struct Work {
    int hq, hkv;
    int m0;      // first query row of the CTA's block, within the sequence
    int rstep;   // Q tile 1 starts rstep rows after Q tile 0 (0 or 128) ...
    int hstep;   // ... in query head hq + hstep (1 when two heads share the rows)
    int lq, lk;  // query / key length of this problem
    int zq, zk;  // TMA coordinates: dense = head slab (b*H + h), varlen = first token
    int q0;      // varlen: first query token of the sequence
    int b;       // dense batch index
    int nk;      // number of KV tiles this block visits (0: every row is empty)
    int kf;      // first KV tile it visits (key windows skip the tiles before it)
};

// Tile order (FlashAttention-4: Blackwell Attention Kernel Co-Design, "LPT scheduling for imbalanced grids"):
// batches (or sequences, longest first) outermost; KV heads in L2-sized
// sections; inside a section the 256-row blocks in reverse order when causal
// (longest work first), then the KV head, then the query heads sharing it.
// The host launches a dense batch as B = 1 with B*Hq query heads over B*Hkv
// KV heads (ALiBi excepted), so one longest-first list covers all of it.
template <bool CAUSAL, bool VARLEN, int VAR>
__device__ __forceinline__ Work decode_tile(const FwdParams& p, uint32_t sched_smem, int t)
{
    Work w;
    int rem = t, nmb;
    w.b = 0;
    w.q0 = 0;
    int k0 = 0;
    // Paired heads: two query heads of one KV head over the same 128 rows, so
    // that under a causal mask both Q tiles see exactly the same keys (256 rows
    // of one head leave the first Q tile a fully masked last KV step).
    const bool pair = CAUSAL && p.pair_heads != 0;
    const int tile_rows = pair ? kBlockM : kRowsPerCta;
    if constexpr (VARLEN) {
        const VarSchedView vs{p, sched_smem};
        int lo = 0, hi = vs.n() - 1;
        while (lo < hi) {  // largest rank whose prefix is <= t
            const int mid = (lo + hi + 1) >> 1;
            if (vs.prefix(mid) <= t) lo = mid;
            else hi = mid - 1;
        }
        const int s = vs.order(lo);
        rem = t - vs.prefix(lo);
        w.q0 = __ldg(p.cu_q + s);
        k0 = __ldg(p.cu_k + s);
        w.lq = __ldg(p.cu_q + s + 1) - w.q0;
        w.lk = __ldg(p.cu_k + s + 1) - k0;
        nmb = (w.lq + tile_rows - 1) / tile_rows;
    } else {
        w.lq = p.Lq;
        w.lk = p.Lk;
        nmb = (p.Lq + tile_rows - 1) / tile_rows;
        const int per_b = nmb * (pair ? (p.Hq >> 1) : p.Hq);
        w.b = t / per_b;
        rem = t - w.b * per_b;
    }
    const int G = p.group, hs = p.heads_per_section;
    const int PG = pair ? (G >> 1) : G;  // query-head slots per KV head
    const int sec_tiles = nmb * hs * PG;
    const int sec = rem / sec_tiles;
    const int rem2 = rem - sec * sec_tiles;
    const int hs_cur = min(hs, p.Hkv - sec * hs);
    const int i = rem2 / (hs_cur * PG);
    const int rem3 = rem2 - i * hs_cur * PG;
    w.hkv = sec * hs + rem3 / PG;
    w.hq = w.hkv * G + (pair ? 2 * (rem3 % PG) : rem3 % PG);
    const int mb = (CAUSAL || (var_window(VAR) && p.desc_tiles)) ? (nmb - 1 - i) : i;
    w.m0 = mb * tile_rows;
    w.rstep = pair ? 0 : kBlockM;
    w.hstep = pair ? 1 : 0;
    if constexpr (VARLEN) {
        w.zq = w.q0;
        w.zk = k0;
    } else {
        w.zq = w.b * p.Hq + w.hq;
        w.zk = w.b * p.Hkv + w.hkv;
    }
    w.kf = 0;
    if (w.lk <= 0) {
        w.nk = 0;
    } else if (var_window(VAR)) {
        // key window [c - left, c + right] around each row's aligned position c
        const int off = w.lk - w.lq;
        const int last_row = min(w.m0 + tile_rows - 1, w.lq - 1);
        const int lo = p.win_left >= 0 ? max(0, w.m0 + off - p.win_left) : 0;
        const int hi = p.win_right >= 0 ? min(w.lk - 1, last_row + off + p.win_right) : w.lk - 1;
        if (hi < lo) {
            w.nk = 0;
        } else {
            w.kf = lo / kBlockN;
            w.nk = hi / kBlockN - w.kf + 1;
        }
    } else if (!CAUSAL) {
        w.nk = (w.lk + kBlockN - 1) / kBlockN;
    } else {
        const int last_row = min(w.m0 + tile_rows - 1, w.lq - 1);
        const int last_key = min(w.lk - 1, last_row + (w.lk - w.lq));
        w.nk = last_key < 0 ? 0 : last_key / kBlockN + 1;
    }
    return w;
}

// The k-th work tile of this CTA.  The persistent grid takes the tile list in
// rounds of gridDim.x.  When tiles differ in length (causal, packed batches,
// key windows) the direction alternates from round to round: with the list
// longest first, a CTA that gets a long tile in one round gets a short one in
// the next (a plain stride leaves the first CTAs 14 % more work than the
// average on a causal 16K sequence).  Equal tiles keep the plain stride, whose
// CTA-to-head placement measured 2 % faster.
template <bool ALTERNATE>
__device__ __forceinline__ int cta_tile(int k)
{
    const int g = (int)gridDim.x;
    return k * g + ((ALTERNATE && (k & 1)) ? g - 1 - (int)blockIdx.x : (int)blockIdx.x);
}

// Two fp32 values to two e4m3 codes (round to nearest even, saturating), `lo`
// in the low byte; and back to fp32.
__device__ __forceinline__ uint16_t e4m3x2_pack(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float2 e4m3x2_unpack(uint16_t v)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    return __half22float2(*reinterpret_cast<__half2*>(&h2));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// All 32 lanes wait on the same barrier; the outcome is made warp-uniform so
// that warp-collective tensor-memory instructions stay aligned.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          const WaitFailure& wf, int site, int tile)
{
    const bool ok = mbar_wait(bar, parity, abort_flag, wf, site, tile);
    return __all_sync(0xffffffffu, ok);
}

// Three barrier phases tested by back-to-back try_waits of one thread (all
// lanes execute it, so the warp stays converged): the three shared-memory
// round trips overlap.  True when all three phases have completed.
__device__ __forceinline__ bool mbar_try_wait3(uint32_t b0, uint32_t p0, uint32_t b1, uint32_t p1, uint32_t b2,
                                               uint32_t p2)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred q0, q1, q2;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 q2, [%5], %6;\n\t"
        "and.pred q0, q0, q1;\n\t"
        "and.pred q0, q0, q2;\n\t"
        "selp.u32 %0, 1, 0, q0;\n\t}\n"
        : "=r"(ok)
        : "r"(b0), "r"(p0), "r"(b1), "r"(p1), "r"(b2), "r"(p2)
        : "memory");
    return ok != 0;
}

// MMA issue sequences of one 128 x 128 x D tile product, executed by the whole
// (converged) MMA warp with lane 0 issuing.  Operands computed in converged
// code stay warp-uniform, and the k-loops are fully unrolled, so tcgen05.mma
// issues back to back (one 128x128x16 MMA per 64 cycles); a rolled loop, or
// operands computed by a single lane, leave the tensor pipe idle between MMAs.
// A descriptor advanced by a byte offset is the base descriptor plus
// offset >> 4 (shared addresses stay below 256 KB, so the field never carries).

// MMA with both operands e4m3 in shared memory (kind::f8f6f4, 32 elements of K).
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor, kind::f8f6f4 with e4m3 A/B (format code 0), fp32 D,
// both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N)
{
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// S_t = Q_t K^T: both operands K-major with 128-byte swizzle, 32 bytes of the
// row (16 bf16 or 32 e4m3 elements) per MMA.  K's first DV columns sit in
// ring stage ks, the rest (D > DV) in tail stage ts.
template <int D, int VAR, int DV>
__device__ __forceinline__ void mma_qk(uint32_t tmem, uint32_t sb, int t, int ks, int ts, bool leader)
{
    using L = FwdSmem<D, VAR, DV>;
    constexpr int kSteps = L::kQBytes / kBlockM / 32;
    constexpr int kMainSteps = L::kTileBytes / kBlockN / 32;
    const uint64_t qd = smem_desc_sw128(sb + L::kQOff + (uint32_t)(t * L::kQBytes), 16, 1024);
    const uint64_t kd = smem_desc_sw128(sb + L::kKVOff + (uint32_t)(ks * L::kTileBytes), 16, 1024);
    const uint64_t td =
        L::kTail ? smem_desc_sw128(sb + L::kTailOff + (uint32_t)(ts * L::kTailBytes), 16, 1024) : 0ull;
    const uint32_t d = tmem + L::kColS + (uint32_t)(t * kBlockN);
    if (leader) {
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk) {
            const uint64_t qoff = (uint64_t)(((kk >> 2) * L::kBlk + (kk & 3) * 32) >> 4);
            const int k2 = kk < kMainSteps ? kk : kk - kMainSteps;
            const uint64_t kdesc = (kk < kMainSteps ? kd : td) + (uint64_t)(((k2 >> 2) * L::kBlk + (k2 & 3) * 32) >> 4);
            if constexpr (L::kFp8)
                mma_ss_f8(d, qd + qoff, kdesc, idesc_e4m3_f32(kBlockM, kBlockN), kk > 0 ? 1u : 0u);
            else
                mma_ss(d, qd + qoff, kdesc, idesc_bf16_f32(kBlockM, kBlockN, false), kk > 0 ? 1u : 0u);
        }
    }
    __syncwarp();
}

// O_t (+)= P_t V.  bf16: P from tensor memory, V MN-major with 128-byte
// swizzle, 16 keys per MMA.  e4m3: P from shared memory (K-major) and V^T
// (K-major, [d][key]), 32 keys per MMA.
template <int D, int VAR, int DV>
__device__ __forceinline__ void mma_pv(uint32_t tmem, uint32_t sb, int t, int vs, bool acc, bool leader)
{
    using L = FwdSmem<D, VAR, DV>;
    const uint32_t d = tmem + L::kColO + (uint32_t)(t * DV);
    if constexpr (L::kFp8) {
        const uint64_t pd = smem_desc_sw128(sb + L::kPOff + (uint32_t)(t * L::kTileBytes), 16, 1024);
        const uint64_t vd = smem_desc_sw128(sb + L::kKVOff + (uint32_t)(vs * L::kTileBytes), 16, 1024);
        if (leader) {
#pragma unroll
            for (int kk = 0; kk < kBlockN / 32; ++kk)
                mma_ss_f8(d, pd + (uint64_t)((kk * 32) >> 4), vd + (uint64_t)((kk * 32) >> 4),
                          idesc_e4m3_f32(kBlockM, DV), (acc || kk > 0) ? 1u : 0u);
        }
    } else {
        constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlockM, DV, true);
        const uint64_t vd = smem_desc_sw128(sb + L::kKVOff + (uint32_t)(vs * L::kTileBytes), L::kBlk, 1024);
        const uint32_t pa = tmem + L::kColP + (uint32_t)t * L::kPStride;
        if (leader) {
#pragma unroll
            for (int kk = 0; kk < kBlockN / 16; ++kk)
                mma_ts(d, pa + (uint32_t)(kk * 8), vd + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV,
                       (acc || kk > 0) ? 1u : 0u);
        }
    }
    __syncwarp();
}

template <int D, bool CAUSAL, bool VARLEN, int VAR, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_sm103_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const FwdParams p)
{
    using L = FwdSmem<D, VAR, DV>;
    constexpr bool kAlternate = CAUSAL || VARLEN || var_window(VAR);  // tiles of unequal length
    // Registers per thread after the split: kSmRegs for the eight softmax
    // warps, kEpiRegs for the four epilogue warps and kCtlRegs for the
    // producer, MMA and two idle warps, 8 * kSmRegs + 4 * (kEpiRegs + kCtlRegs)
    // = 16 * 128, the launch's own count.  Measured per kernel (ptxas spills
    // move between the roles with the split): with D >= 128 a packed batch's
    // epilogue spilled at 64 (addresses through the sequence offsets), and
    // 192 / 80 / 48 took the 8-sequence causal workload from 1.293 to
    // 1.256 ms; the plain dense D = 128 kernel ran 1 % faster at
    // 184 / 80 / 64; the causal dense kernel ran best at 192 / 64 / 64 (3 %
    // slower with either of the others).
    constexpr bool kPlainDense = !CAUSAL && !VARLEN && VAR == kVarNone && D == 128 && DV == 128;
    constexpr int kSmRegs = kPlainDense ? 184 : 192;
    constexpr int kEpiRegs = (kPlainDense || (VARLEN && D >= 128)) ? 80 : 64;
    constexpr int kCtlRegs = 512 - 2 * kSmRegs - kEpiRegs;
    static_assert(kCtlRegs >= 40 && kSmRegs % 8 == 0 && kEpiRegs % 8 == 0 && kCtlRegs % 8 == 0,
                  "setmaxnreg split must fill the launch's 16 x 128 registers per lane");
    constexpr bool kSoftmaxFreesKV = !L::kTail && !L::kFp8;  // who frees K/V ring stages (see the softmax role)
    constexpr float kTau = 8.0f;     // rescale threshold, log2 units
    constexpr float kLn2 = 0.69314718055994530942f;

    // operand tiles need 1 KB alignment of their shared-memory address (the
    // 128-byte swizzle pattern repeats every 8 rows of 128 bytes)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + L::kBarOff;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
    float2* stats = reinterpret_cast<float2*>(smem + L::kStatsOff);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WaitFailure wf{p.err, p.diag};
    using SS = FwdSchedSmem<D, VAR, DV>;
    constexpr int kUsed = VARLEN ? SS::kBytes : L::kBytes;
    if ((uint32_t)(smem - smem_raw) + kUsed > (uint32_t)fwd_smem_alloc<D, VARLEN, VAR, DV>()) {
        // the dynamic window is aligned too loosely for the layout: report, touch nothing
        if (threadIdx.x == 0) atomicOr(p.err, 4);
        return;
    }

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(L::kQFull + t), 1);
            mbar_init(bar(L::kQEmpty + t), 1);
            mbar_init(bar(L::kSFull + t), 1);
            mbar_init(bar(L::kPFull + t), kBlockM);
            mbar_init(bar(L::kOFull + t), 1);
            mbar_init(bar(L::kOEmpty + t), kBlockM);
            mbar_init(bar(L::kStFull + t), kBlockM);
            mbar_init(bar(L::kStEmpty + t), kBlockM);
            mbar_init(bar(L::kSEmpty + t), kBlockM);
            mbar_init(bar(L::kPEmpty + t), 1);
        }
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(bar(L::kKVFull + s), 1);
            mbar_init(bar(L::kKVEmpty + s), L::kSplitP ? 2 : 1);  // split P: one arrival per Q tile
        }
        for (int s = 0; s < L::kTailStages; ++s) {
            mbar_init(bar(L::kTFull + s), 1);
            mbar_init(bar(L::kTEmpty + s), 1);
        }
        mbar_init(bar(L::kDrain), L::kSplitP ? 2 : 1);  // split P: both MMA warps
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 12 && lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
    }
    if (warp == 13) {
        tmem_alloc(smem_u32(tmem_slot), L::kTmemCols);
        tmem_relinquish();
    }
    if (VARLEN && !p.sched) {
        int* prefix = reinterpret_cast<int*>(smem + SS::kOff);
        int* order = prefix + p.seq_count + 1;
        auto* keys = reinterpret_cast<unsigned long long*>(smem + L::kKVOff);
        build_varlen_schedule<SS::kPad>(p, keys, reinterpret_cast<int*>(keys + SS::kPad), prefix, order);
        // the sort's generic-proxy writes to the ring precede the TMA writes into it
        fence_proxy_async_shared();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    int num_tiles = p.num_tiles;
    if constexpr (VARLEN) {
        const VarSchedView vs{p, sb + SS::kOff};
        num_tiles = vs.prefix(vs.n());
    }

    if (warp < 8) {
        // ============================================================ softmax
        regs_increase<kSmRegs>();
        const int t = warp >> 2;             // Q tile of this group
        const int row = threadIdx.x & 127;   // query row within the tile == TMEM lane
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t tS = tmem + lane_base + L::kColS + (uint32_t)(t * kBlockN);
        const uint32_t tP = tmem + lane_base + L::kColP + (uint32_t)t * L::kPStride;
        const uint32_t tO = tmem + lane_base + L::kColO + (uint32_t)(t * DV);
        const float sl2 = p.scale_log2;
        uint32_t s_ph = 0, st_ph = 1;
        uint32_t pe_ph = 0;      // split P: phase of the P.V-done barrier
        bool p_written = false;  // split P: a P of this group is in tensor memory
        // K/V ring slots taken before the current work tile (K(0), V(0), K(1), ...)
        uint32_t kv_seq = 0;
        // The first thread of the tile-1 group frees the K/V stages (a commit
        // costs the MMA warp about 100 cycles of tensor-pipe idle time): S1(j)
        // complete means every MMA issued before it has completed -- S0(j),
        // P0(j-1).V(j-1) and P1(j-1).V(j-1) -- so K(j) and V(j-1) are no longer
        // read.  (The MMA warp frees the last V of a work tile.)  A three-stage
        // ring (D > DV) cannot wait that long for V(j-1), and with e4m3 operands
        // the softmax, not the MMA warp, bounds the step: in both the MMA warp
        // commits every release as soon as the MMAs reading the stage are issued.
        // With P in columns of its own the next S is issued before this step's
        // P.V, so V(j-1) is freed only once P1(j-1).V(j-1) has completed (the
        // group waits for that before it overwrites P1).
        // With P in columns of its own each Q tile has its own MMA warp, so each
        // group's first thread frees its share (the barriers count two arrivals):
        // K(j) once S_t(j) has completed, V(j-1) once P_t(j-1).V(j-1) has.
        const bool kv_releaser = kSoftmaxFreesKV && (L::kSplitP || t == 1) && row == 0;
        for (int k = 0, tile = cta_tile<kAlternate>(0); tile < num_tiles; tile = cta_tile<kAlternate>(++k)) {
            const Work w = decode_tile<CAUSAL, VARLEN, VAR>(p, sb + SS::kOff, tile);
            if (w.nk == 0) continue;
            const int q_row = w.m0 + t * w.rstep + row;
            const int hq_t = w.hq + t * w.hstep;  // query head of this Q tile
            int kv_last = w.lk - 1;  // last key this row may attend
            int kv_first = 0;        // first key this row may attend
            const int c_row = q_row + (w.lk - w.lq);  // the row's aligned position among the keys
            if (CAUSAL) kv_last = min(kv_last, c_row);
            if constexpr (var_window(VAR)) {
                if (p.win_right >= 0) kv_last = min(kv_last, c_row + p.win_right);
                if (p.win_left >= 0) kv_first = max(0, c_row - p.win_left);
            }
            float alibi_l2 = 0.f;  // ALiBi slope of this head, log2 units
            if constexpr (var_alibi(VAR)) alibi_l2 = __ldg(p.alibi + hq_t) * 1.4426950408889634f;
            // score multiplier inside the exponent: the score modifiers already
            // produce log2-unit scores; e4m3 scores carry the tiles' scales
            constexpr bool kLog2Mod = var_softcap(VAR) || var_alibi(VAR);
            float smul = kLog2Mod ? 1.f : sl2;
            const float* fp8_sk = nullptr;
            if constexpr (VAR == kVarFp8) {
                smul = sl2 * __ldg(p.fp8_sq + ((long long)w.b * p.Hq + hq_t) * p.fp8_nq + (w.m0 + t * w.rstep) / kBlockM);
                fp8_sk = p.fp8_sk + ((long long)w.b * p.Hkv + w.hkv) * p.fp8_nk + w.kf;
            }
            const float smul_q = smul;
            // r: reference; l: sum of the fp32 p; l_rnd: e4m3 P -- sum of the rounded
            // p, bf16 P -- sum of the rounding errors of each step's largest p
            float r = -INFINITY, l = 0.f, l_rnd = 0.f;
            for (int j = 0; j < w.nk; ++j) {
                if (!warp_wait(bar(L::kSFull + t), s_ph, abort_flag, wf, 1 + t, tile)) goto done;
                s_ph ^= 1;
                if (kv_releaser) {
                    mbar_arrive(bar(L::kKVEmpty + (int)((kv_seq + 2u * (uint32_t)j) % (uint32_t)L::kStages)));
                    if (!L::kSplitP && j > 0)
                        mbar_arrive(bar(L::kKVEmpty + (int)((kv_seq + 2u * (uint32_t)j - 1u) % (uint32_t)L::kStages)));
                }
                tc_fence_after_sync();
                uint32_t sv[4][32];
                // the tensor-memory load also returns each chunk's maximum when the
                // raw score order is the order the row maximum needs
                constexpr bool kHwMax = VAR == kVarNone || VAR == kVarWindow || VAR == kVarFp8;
                float hmx[4] = {0.f, 0.f, 0.f, 0.f};  // set by the loads when kHwMax
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if constexpr (kHwMax)
                        tmem_ld32_max(tS + 32u * c, sv[c], hmx[c]);
                    else
                        tmem_ld32(tS + 32u * c, sv[c]);
                }
                tmem_wait_ld();
                if constexpr (L::kSplitP) {
                    // S is in registers: its columns may take the next S
                    tc_fence_before_sync();
                    mbar_arrive(bar(L::kSEmpty + t));
                }
                const int key0 = (j + w.kf) * kBlockN;
                if constexpr (VAR == kVarFp8) smul = smul_q * __ldg(fp8_sk + j);
                // score modifiers (FlashAttention from Scratch, sec. 12), in log2 units:
                // soft-capping of the scaled score, then the ALiBi distance bias
                if constexpr (var_softcap(VAR)) {
                    // cap * tanh(s * scale / cap), tanh(u) = 1 - 2 / (1 + e^(2u))
                    const float k2 = p.cap_in * (2.f * 1.4426950408889634f);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const float e2u = ex2_approx(__uint_as_float(sv[c][i]) * k2);
                            const float th = fmaf(-2.f, rcp_approx(1.f + e2u), 1.f);
                            sv[c][i] = __float_as_uint(th * p.cap_out);
                        }
                }
                if constexpr (var_alibi(VAR)) {
                    // s' - slope * |c - key|, s' = s * scale or the capped score
                    const float cf = (float)(c_row - key0);
                    const float pre = var_softcap(VAR) ? 1.f : sl2;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            sv[c][i] = __float_as_uint(fmaf(-alibi_l2, fabsf(cf - (float)(32 * c + i)),
                                                            __uint_as_float(sv[c][i]) * pre));
                }
                // masking: keys outside [kv_first, kv_last] (causal diagonal, key
                // window, sequence tail) get -inf (FlashAttention from Scratch, sec. 7.3)
                const int nvalid = kv_last - key0 + 1;
                const int nskip = kv_first - key0;
                const bool masked = __any_sync(0xffffffffu, nvalid < kBlockN || nskip > 0);
                if (masked) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (32 * c + i >= nvalid || 32 * c + i < nskip) sv[c][i] = __float_as_uint(-INFINITY);
                }
                // row maximum of the scores: from the loads, unless masking or a
                // score modifier changed the values
                float mraw;
                if (kHwMax && !masked) {
                    mraw = fmaxf(fmaxf(hmx[0], hmx[1]), fmaxf(hmx[2], hmx[3]));
                } else {
                    float mx[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mx[i] = __uint_as_float(sv[i >> 1][(i & 1) * 16]);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int e = 32 * c + i;
                            if ((e & 15) == 0) continue;
                            mx[e >> 4] = fmaxf(mx[e >> 4], __uint_as_float(sv[c][i]));
                        }
#pragma unroll
                    for (int i = 0; i < 4; ++i) mx[i] = fmaxf(mx[i], mx[i + 4]);
                    mraw = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                }
                const float mrow = mraw * smul;
                // conditional rescale: keep r unless the maximum rose by more than tau
                const float r_new = (mrow - r > kTau) ? mrow : r;
                const float alpha = (r_new == r) ? 1.f : ex2_approx(r - r_new);
                const float r_use = (r_new == -INFINITY) ? 0.f : r_new;
                l *= alpha;
                // p = 2^(s*scale*log2e - r), rounded to bf16 (e4m3) for the P.V MMA.
                // The sum of the fp32 p gives the LSE.  O is normalised by the sum of
                // the ROUNDED p, so that numerator and denominator weight every key
                // alike (a row dominated by one key would otherwise err by up to
                // |v| * 2^-9).  For bf16 P that sum is taken as the fp32 sum plus the
                // rounding error of each step's largest p -- the key that can
                // dominate -- computed once from the step maximum with the same
                // fused multiply-add, exponential and rounding as its element; the
                // other keys' rounding errors average out over the row.  For e4m3 P
                // (3-bit mantissa) the rounded values are summed in full.
                l_rnd *= alpha;
                const uint64_t c2 = f2_pack(smul, smul);
                const uint64_t nr2 = f2_pack(-r_use, -r_use);
                uint64_t sum_t[2] = {0ull, 0ull}, sum_r[2] = {0ull, 0ull};
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = 64 * c + 2 * i;
                        const uint64_t x2 = f2_fma(f2_pack(__uint_as_float(sv[e >> 5][e & 31]),
                                                           __uint_as_float(sv[(e + 1) >> 5][(e + 1) & 31])),
                                                   c2, nr2);
                        float x0, x1;
                        f2_unpack(x2, x0, x1);
                        const float e0 = ex2_approx(x0), e1 = ex2_approx(x1);
                        sum_t[i & 1] = f2_add(sum_t[i & 1], f2_pack(e0, e1));
                        if constexpr (VAR == kVarFp8) {
                            const uint16_t h = e4m3x2_pack(e0, e1);
                            const float2 rf = e4m3x2_unpack(h);
                            sum_r[i & 1] = f2_add(sum_r[i & 1], f2_pack(rf.x, rf.y));
                            if (i & 1)
                                pk[i >> 1] |= (uint32_t)h << 16;
                            else
                                pk[i >> 1] = h;
                        } else {
                            pk[i] = pack_bf16x2(e0, e1);
                        }
                    }
                    if constexpr (VAR == kVarFp8) {
                        // P (e4m3, keys 64c .. 64c+63 = 16-byte chunks 4c .. 4c+3 of the
                        // row) into the P tile, 128-byte swizzle, for the SS P.V MMA
                        const uint32_t prow = sb + L::kPOff + (uint32_t)(t * L::kTileBytes + row * 128);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            st_shared_v4(prow + (uint32_t)(((4 * c + u) ^ (row & 7)) << 4), pk[4 * u], pk[4 * u + 1],
                                         pk[4 * u + 2], pk[4 * u + 3]);
                    } else {
                        if constexpr (L::kSplitP) {
                            if (c == 0) {
                                // the last P.V of this group has read P (and, for the
                                // tile-1 group, V(j-1)) and left O idle
                                if (p_written) {
                                    if (!warp_wait(bar(L::kPEmpty + t), pe_ph, abort_flag, wf, 27 + t, tile)) goto done;
                                    pe_ph ^= 1;
                                    tc_fence_after_sync();
                                    if (kv_releaser && j > 0)
                                        mbar_arrive(bar(L::kKVEmpty +
                                                        (int)((kv_seq + 2u * (uint32_t)j - 1u) % (uint32_t)L::kStages)));
                                }
                                p_written = true;
                            }
                            tmem_st32(tP + 32u * c, pk);
                        } else {
                            // P (bf16 pairs) over the first 64 columns of S
                            tmem_st32(tS + 32u * c, pk);
                        }
                    }
                }
                if constexpr (VAR == kVarFp8) fence_proxy_async_shared();  // P visible to the tensor core
                {
                    float a0, a1;
                    f2_unpack(f2_add(sum_t[0], sum_t[1]), a0, a1);
                    l += a0 + a1;
                    if constexpr (VAR == kVarFp8) {
                        float b0, b1;
                        f2_unpack(f2_add(sum_r[0], sum_r[1]), b0, b1);
                        l_rnd += b0 + b1;
                    } else {
                        const float pm = ex2_approx(fmaf(mraw, smul, -r_use));  // the step's largest p
                        l_rnd += __uint_as_float(pack_bf16x2(pm, 0.f) << 16) - pm;
                    }
                }
                // correction of the accumulator when the reference moved (O is idle
                // here: the previous P.V completed before this S was committed, or,
                // with P in columns of its own, before the wait above returned)
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    // two 32-column chunks per tensor-memory round trip
#pragma unroll 1
                    for (int c = 0; c < DV / 32; c += 2) {
                        uint32_t ov[2][32];
                        tmem_ld32(tO + 32u * c, ov[0]);
                        tmem_ld32(tO + 32u * (c + 1), ov[1]);
                        tmem_wait_ld();
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) ov[h][i] = __float_as_uint(__uint_as_float(ov[h][i]) * alpha);
                            tmem_st32(tO + 32u * (c + h), ov[h]);
                        }
                    }
                }
                tmem_wait_st();
                tc_fence_before_sync();
                mbar_arrive(bar(L::kPFull + t));
                r = r_new;
            }
            kv_seq += 2u * (uint32_t)w.nk;
            // hand the row statistics to the epilogue
            if (!warp_wait(bar(L::kStEmpty + t), st_ph, abort_flag, wf, 3 + t, tile)) goto done;
            st_ph ^= 1;
            // (sum of rounded p, base-2 log of the row's normaliser)
            const float l_o = VAR == kVarFp8 ? l_rnd : l + l_rnd;
            stats[t * kBlockM + row] = make_float2(l_o, l > 0.f ? r + __log2f(l) : -INFINITY);
            mbar_arrive(bar(L::kStFull + t));
        }
    } else if (warp < 12) {
        // ============================================================ epilogue
        regs_decrease<kEpiRegs>();
        const int row = threadIdx.x & 127;
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        uint32_t o_ph[2] = {0, 0}, st_ph[2] = {0, 0};
        float* obase = reinterpret_cast<float*>(p.o);
        for (int k = 0, tile = cta_tile<kAlternate>(0); tile < num_tiles; tile = cta_tile<kAlternate>(++k)) {
            const Work w = decode_tile<CAUSAL, VARLEN, VAR>(p, sb + SS::kOff, tile);
            for (int t = 0; t < 2; ++t) {
                const int q_row = w.m0 + t * w.rstep + row;
                const int hq_t = w.hq + t * w.hstep;
                const bool valid = q_row < w.lq;
                int64_t orow, lidx;
                if constexpr (VARLEN) {
                    orow = ((int64_t)(w.q0 + q_row) * p.Hq + hq_t) * DV;
                    lidx = (int64_t)hq_t * p.total_q + w.q0 + q_row;
                } else {
                    lidx = ((int64_t)w.b * p.Hq + hq_t) * p.Lq + q_row;
                    orow = lidx * DV;
                }
                uint4* dst = reinterpret_cast<uint4*>(obase + orow);
                if (w.nk == 0) {  // no key reaches this block: O = 0, LSE = -inf
                    if (valid) {
#pragma unroll
                        for (int i = 0; i < DV / 4; ++i) dst[i] = make_uint4(0, 0, 0, 0);
                        p.lse[lidx] = -INFINITY;
                    }
                    continue;
                }
                if (!warp_wait(bar(L::kOFull + t), o_ph[t], abort_flag, wf, 5 + t, tile)) goto done;
                o_ph[t] ^= 1;
                tc_fence_after_sync();
                if (!warp_wait(bar(L::kStFull + t), st_ph[t], abort_flag, wf, 7 + t, tile)) goto done;
                st_ph[t] ^= 1;
                const float2 st = stats[t * kBlockM + row];  // (sum of rounded p, log2 normaliser)
                mbar_arrive(bar(L::kStEmpty + t));
                float inv = st.x > 0.f ? 1.f / st.x : 0.f;
                if constexpr (VAR == kVarFp8) inv *= __ldg(p.fp8_sv + (long long)w.b * p.Hkv + w.hkv);
                const uint32_t tO = tmem + lane_base + L::kColO + (uint32_t)(t * DV);
                if constexpr (L::kEpiStaged) {
                    // Each 32 x 32 block of the warp's rows goes through shared memory:
                    // a thread writes its own row, then every store instruction writes
                    // four whole 128-byte row segments (a thread per row would touch
                    // 32 scattered sectors per instruction).
                    const uint32_t stage = sb + L::kEpiOff + (uint32_t)((warp & 3) * L::kEpiWarpBytes);
                    const int rsub = lane >> 3, cq = lane & 7;  // row within a group of four, 16-byte column
                    const int wrow0 = w.m0 + t * w.rstep + 32 * (warp & 3);
                    const int64_t rstride = VARLEN ? (int64_t)p.Hq * DV : (int64_t)DV;
                    float* wbase = obase + (VARLEN ? ((int64_t)(w.q0 + wrow0) * p.Hq + hq_t) * DV
                                                   : (((int64_t)w.b * p.Hq + hq_t) * p.Lq + wrow0) * DV);
#pragma unroll 1
                    for (int c = 0; c < DV / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(tO + 32u * c, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            st_shared_v4(stage + (uint32_t)(lane * L::kEpiRowBytes + 16 * u),
                                         __float_as_uint(__uint_as_float(ov[4 * u]) * inv),
                                         __float_as_uint(__uint_as_float(ov[4 * u + 1]) * inv),
                                         __float_as_uint(__uint_as_float(ov[4 * u + 2]) * inv),
                                         __float_as_uint(__uint_as_float(ov[4 * u + 3]) * inv));
                        __syncwarp();
#pragma unroll
                        for (int k4 = 0; k4 < 8; ++k4) {
                            const int r = 4 * k4 + rsub;
                            const uint4 v = ld_shared_v4(stage + (uint32_t)(r * L::kEpiRowBytes + 16 * cq));
                            if (wrow0 + r < w.lq)
                                *reinterpret_cast<uint4*>(wbase + r * rstride + 32 * c + 4 * cq) = v;
                        }
                        __syncwarp();
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < DV / 32; ++c) {
                        uint32_t ov[32];
                        tmem_ld32(tO + 32u * c, ov);
                        tmem_wait_ld();
                        if (valid) {
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                dst[8 * c + i] = make_uint4(__float_as_uint(__uint_as_float(ov[4 * i]) * inv),
                                                            __float_as_uint(__uint_as_float(ov[4 * i + 1]) * inv),
                                                            __float_as_uint(__uint_as_float(ov[4 * i + 2]) * inv),
                                                            __float_as_uint(__uint_as_float(ov[4 * i + 3]) * inv));
                        }
                    }
                }
                tc_fence_before_sync();
                mbar_arrive(bar(L::kOEmpty + t));
                if (valid) p.lse[lidx] = st.y * kLn2;
            }
        }
    } else {
        regs_decrease<kCtlRegs>();
        if (warp == 12) {
            // ============================================================ TMA producer
            if (lane == 0) {
                uint32_t q_ph[2] = {1, 1};
                int stage = 0, tstage = 0;
                uint32_t kv_ph = 1, t_ph = 1;
                // last armed phase of each buffer, to wait out copies in flight at exit
                int q_armed[2] = {-1, -1};
                int kv_armed[L::kStages];
                int t_armed[L::kTailStages > 0 ? L::kTailStages : 1];
                for (int s = 0; s < L::kStages; ++s) kv_armed[s] = -1;
                for (int s = 0; s < L::kTailStages; ++s) t_armed[s] = -1;
                auto load_q = [&](const Work& w, int t, int tile) -> bool {
                    if (!mbar_wait(bar(L::kQEmpty + t), q_ph[t], abort_flag, wf, 9 + t, tile)) return false;
                    q_ph[t] ^= 1;
                    mbar_arrive_expect_tx(bar(L::kQFull + t), L::kQBytes);
                    q_armed[t] = (int)q_ph[t];  // parity of the phase this copy completes
                    const uint32_t dst = sb + L::kQOff + (uint32_t)(t * L::kQBytes);
                    const int row0 = w.m0 + t * w.rstep;
#pragma unroll
                    for (int h = 0; h < L::kHalvesQ; ++h) {
                        if constexpr (VARLEN)
                            tma_load_3d(dst + h * L::kBlk, &tmQ, bar(L::kQFull + t), 64 * h, w.hq + t * w.hstep,
                                        w.zq + row0);
                        else
                            tma_load_3d(dst + h * L::kBlk, &tmQ, bar(L::kQFull + t), 64 * h, row0,
                                        w.zq + t * w.hstep);
                    }
                    return true;
                };
                auto load_kv = [&](const CUtensorMap* map, const Work& w, int j, int tile) -> bool {
                    if (!mbar_wait(bar(L::kKVEmpty + stage), kv_ph, abort_flag, wf, 11, tile)) return false;
                    if (p.fault == 1 && j == 0 && map == &tmK && tile == (int)blockIdx.x) {
                        // test hook: this K tile is never armed or loaded, so the wait
                        // for it runs out and the launch reports a timeout
                        if (++stage == L::kStages) {
                            stage = 0;
                            kv_ph ^= 1;
                        }
                        return true;
                    }
                    mbar_arrive_expect_tx(bar(L::kKVFull + stage), L::kTileBytes);
                    kv_armed[stage] = (int)(kv_ph ^ 1u);
                    const uint32_t dst = sb + L::kKVOff + (uint32_t)(stage * L::kTileBytes);
                    if (L::kFp8 && map == &tmV) {
                        // e4m3 V is stored transposed, [d][key]: the tile is keys
                        // (j+kf)*128 .. +127 of all 128 rows d
                        tma_load_3d(dst, map, bar(L::kKVFull + stage), (j + w.kf) * kBlockN, 0, w.zk);
                    } else {
#pragma unroll
                        for (int h = 0; h < L::kHalves; ++h) {
                            if constexpr (VARLEN)
                                tma_load_3d(dst + h * L::kBlk, map, bar(L::kKVFull + stage), 64 * h, w.hkv,
                                            w.zk + (j + w.kf) * kBlockN);
                            else
                                tma_load_3d(dst + h * L::kBlk, map, bar(L::kKVFull + stage), 64 * h,
                                            (j + w.kf) * kBlockN, w.zk);
                        }
                    }
                    if (++stage == L::kStages) {
                        stage = 0;
                        kv_ph ^= 1;
                    }
                    if (L::kTail && map == &tmK) {
                        // K columns DV .. D-1 into the tail ring
                        if (!mbar_wait(bar(L::kTEmpty + tstage), t_ph, abort_flag, wf, 24, tile)) return false;
                        mbar_arrive_expect_tx(bar(L::kTFull + tstage), L::kTailBytes);
                        t_armed[tstage] = (int)(t_ph ^ 1u);
                        const uint32_t tdst = sb + L::kTailOff + (uint32_t)(tstage * L::kTailBytes);
#pragma unroll
                        for (int h = 0; h < L::kTailHalves; ++h) {
                            if constexpr (VARLEN)
                                tma_load_3d(tdst + h * L::kBlk, map, bar(L::kTFull + tstage), 64 * (L::kHalves + h),
                                            w.hkv, w.zk + (j + w.kf) * kBlockN);
                            else
                                tma_load_3d(tdst + h * L::kBlk, map, bar(L::kTFull + tstage), 64 * (L::kHalves + h),
                                            (j + w.kf) * kBlockN, w.zk);
                        }
                        if (++tstage == L::kTailStages) {
                            tstage = 0;
                            t_ph ^= 1;
                        }
                    }
                    return true;
                };
                for (int k = 0, tile = cta_tile<kAlternate>(0); tile < num_tiles; tile = cta_tile<kAlternate>(++k)) {
                    const Work w = decode_tile<CAUSAL, VARLEN, VAR>(p, sb + SS::kOff, tile);
                    if (w.nk == 0) continue;
                    if (!load_q(w, 0, tile)) break;
                    if (!load_kv(&tmK, w, 0, tile)) break;
                    if (!load_q(w, 1, tile)) break;
                    if (!load_kv(&tmV, w, 0, tile)) break;
                    bool ok = true;
                    for (int j = 1; j < w.nk && ok; ++j) ok = load_kv(&tmK, w, j, tile) && load_kv(&tmV, w, j, tile);
                    if (!ok) break;
                }
                // every copy this warp started has landed before the CTA retires
                for (int t = 0; t < 2; ++t)
                    if (q_armed[t] >= 0) mbar_settle(bar(L::kQFull + t), (uint32_t)q_armed[t], wf, 13);
                for (int s = 0; s < L::kStages; ++s)
                    if (kv_armed[s] >= 0) mbar_settle(bar(L::kKVFull + s), (uint32_t)kv_armed[s], wf, 14);
                for (int s = 0; s < L::kTailStages; ++s)
                    if (t_armed[s] >= 0) mbar_settle(bar(L::kTFull + s), (uint32_t)t_armed[s], wf, 26);
            }
            __syncwarp();
        } else if (warp == 13 || (L::kSplitP && warp == 14)) {
            // ============================================================ MMA issuer
            // The whole warp runs this loop; lane 0 issues every MMA and commit (a
            // commit tracks the MMAs of the thread that executes it).
            const bool leader = lane == 0;
            const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
            uint32_t q_ph[2] = {0, 0}, p_ph[2] = {0, 0}, oe_ph[2] = {1, 1};
            int stage = 0, tstage = 0;
            uint32_t kv_ph = 0, t_ph = 0;
            bool issued = false;
            auto next_stage = [&]() {
                if (++stage == L::kStages) {
                    stage = 0;
                    kv_ph ^= 1;
                }
            };
            auto commit = [&](int b) {
                if (leader) tc_commit(bar(b));
                __syncwarp();
            };
            // the tail stage of the K tile just taken from the ring (D > DV only)
            auto take_tail = [&](int tile, int& ts) -> bool {
                ts = 0;
                if constexpr (L::kTail) {
                    ts = tstage;
                    if (!warp_wait(bar(L::kTFull + ts), t_ph, abort_flag, wf, 25, tile)) return false;
                    if (++tstage == L::kTailStages) {
                        tstage = 0;
                        t_ph ^= 1;
                    }
                }
                return true;
            };
            auto release_tail = [&](int ts) {
                if constexpr (L::kTail) commit(L::kTEmpty + ts);
            };
            if constexpr (L::kSplitP) {
                // P in columns of its own, one MMA warp per Q tile (warp 13: tile 0,
                // warp 14: tile 1; the tensor pipe interleaves their MMAs).  Per KV
                // step j the warp issues S_t(j+1) as soon as its softmax group has
                // read S_t(j) (and K(j+1) has landed), then P_t(j).V(j) when P
                // arrives, so the group's next scores are ready while it is still on
                // the exponentials, and neither group waits for the other's MMAs.
                // Ring slots are numbered from the start of the launch: K(j) of a
                // work tile is kv_base + 2j, V(j) kv_base + 2j + 1.
                const int t = warp - 13;
                uint32_t se_ph = 0;
                uint32_t kv_base = 0;
                bool s_any = false;  // an S has been issued (later ones wait for the softmax to read it)
                auto slot_wait = [&](uint32_t slot, int site, int tile) -> bool {
                    return warp_wait(bar(L::kKVFull + (int)(slot % (uint32_t)L::kStages)),
                                     (slot / (uint32_t)L::kStages) & 1u, abort_flag, wf, site, tile);
                };
                // S_t into its columns from K in ring slot kslot
                auto issue_s = [&](uint32_t kslot, int tile) -> bool {
                    if (s_any) {
                        if (!warp_wait(bar(L::kSEmpty + t), se_ph, abort_flag, wf, 29 + t, tile)) return false;
                        se_ph ^= 1;
                    }
                    s_any = true;
                    tc_fence_after_sync();
                    mma_qk<D, VAR, DV>(tm, sb, t, (int)(kslot % (uint32_t)L::kStages), 0, leader);
                    issued = true;
                    commit(L::kSFull + t);
                    return true;
                };
                for (int k = 0, tile = cta_tile<kAlternate>(0); tile < num_tiles; tile = cta_tile<kAlternate>(++k)) {
                    const Work w = decode_tile<CAUSAL, VARLEN, VAR>(p, sb + SS::kOff, tile);
                    if (w.nk == 0) continue;
                    const int nk = w.nk;
                    bool ok = warp_wait(bar(L::kQFull + t), q_ph[t], abort_flag, wf, 15 + t, tile) &&
                              slot_wait(kv_base, 17, tile) && issue_s(kv_base, tile);
                    q_ph[t] ^= 1;
                    if (ok && nk == 1) commit(L::kQEmpty + t);
                    for (int j = 0; j < nk && ok; ++j) {
                        const bool last = j + 1 == nk;
                        if (!last) {
                            const uint32_t ks = kv_base + 2u * (uint32_t)(j + 1);
                            if (!(ok = slot_wait(ks, 17, tile) && issue_s(ks, tile))) break;
                            if (j + 2 == nk) commit(L::kQEmpty + t);
                        }
                        const uint32_t vslot = kv_base + 2u * (uint32_t)j + 1u;
                        if (!(ok = slot_wait(vslot, 18, tile))) break;
                        if (j == 0) {
                            if (!(ok = warp_wait(bar(L::kOEmpty + t), oe_ph[t], abort_flag, wf, 19 + t, tile))) break;
                            oe_ph[t] ^= 1;
                        }
                        if (!(ok = warp_wait(bar(L::kPFull + t), p_ph[t], abort_flag, wf, 21 + t, tile))) break;
                        p_ph[t] ^= 1;
                        tc_fence_after_sync();
                        const int vs = (int)(vslot % (uint32_t)L::kStages);
                        mma_pv<D, VAR, DV>(tm, sb, t, vs, j > 0, leader);
                        commit(L::kPEmpty + t);
                        if (last) {
                            commit(L::kOFull + t);
                            commit(L::kKVEmpty + vs);  // this tile's share of the last V
                        }
                    }
                    if (!ok) break;
                    kv_base += 2u * (uint32_t)nk;
                }
            } else {
                for (int k = 0, tile = cta_tile<kAlternate>(0); tile < num_tiles; tile = cta_tile<kAlternate>(++k)) {
                    const Work w = decode_tile<CAUSAL, VARLEN, VAR>(p, sb + SS::kOff, tile);
                    if (w.nk == 0) continue;
                    const int nk = w.nk;
                    // prologue: S0(0), S1(0)
                    if (!warp_wait(bar(L::kQFull + 0), q_ph[0], abort_flag, wf, 15, tile)) break;
                    q_ph[0] ^= 1;
                    const int ks = stage;
                    if (!warp_wait(bar(L::kKVFull + ks), kv_ph, abort_flag, wf, 17, tile)) break;
                    next_stage();
                    int ts;
                    if (!take_tail(tile, ts)) break;
                    tc_fence_after_sync();
                    mma_qk<D, VAR, DV>(tm, sb, 0, ks, ts, leader);
                    issued = true;
                    commit(L::kSFull + 0);
                    if (nk == 1) commit(L::kQEmpty + 0);
                    if (!warp_wait(bar(L::kQFull + 1), q_ph[1], abort_flag, wf, 16, tile)) break;
                    q_ph[1] ^= 1;
                    tc_fence_after_sync();
                    mma_qk<D, VAR, DV>(tm, sb, 1, ks, ts, leader);
                    commit(L::kSFull + 1);
                    if constexpr (!kSoftmaxFreesKV) commit(L::kKVEmpty + ks);
                    release_tail(ts);
                    if (nk == 1) commit(L::kQEmpty + 1);
                    bool ok = true;
                    for (int j = 0; j < nk && ok; ++j) {
                        // V(j), K(j+1) and P0(j): in the steady state all three have
                        // completed when the warp gets here, and one combined test costs one
                        // shared-memory round trip; otherwise they are awaited one by one
                        const int vs = stage;
                        const uint32_t vph = kv_ph;
                        next_stage();
                        int kn = -1, tn = 0;
                        uint32_t kph = vph;
                        if (j + 1 < nk) {
                            kn = stage;
                            kph = kv_ph;
                            next_stage();
                        }
                        const bool all3 = j > 0 &&
                            __all_sync(0xffffffffu, mbar_try_wait3(bar(L::kKVFull + vs), vph,
                                                                   bar(L::kKVFull + (kn >= 0 ? kn : vs)), kph,
                                                                   bar(L::kPFull + 0), p_ph[0]));
                        if (!all3) {
                            if (!(ok = warp_wait(bar(L::kKVFull + vs), vph, abort_flag, wf, 18, tile))) break;
                            if (kn >= 0 && !(ok = warp_wait(bar(L::kKVFull + kn), kph, abort_flag, wf, 17, tile))) break;
                        }
                        if (kn >= 0 && !(ok = take_tail(tile, tn))) break;
                        // tile 0: P0(j) . V(j), then S0(j+1)
                        if (j == 0) {
                            if (!(ok = warp_wait(bar(L::kOEmpty + 0), oe_ph[0], abort_flag, wf, 19, tile))) break;
                            oe_ph[0] ^= 1;
                        }
                        if (!all3 && !(ok = warp_wait(bar(L::kPFull + 0), p_ph[0], abort_flag, wf, 21, tile))) break;
                        p_ph[0] ^= 1;
                        tc_fence_after_sync();
                        mma_pv<D, VAR, DV>(tm, sb, 0, vs, j > 0, leader);
                        if (kn >= 0) {
                            mma_qk<D, VAR, DV>(tm, sb, 0, kn, tn, leader);
                            commit(L::kSFull + 0);
                            if (j + 2 == nk) commit(L::kQEmpty + 0);
                        } else {
                            commit(L::kOFull + 0);
                        }
                        // tile 1: P1(j) . V(j), then S1(j+1)
                        if (j == 0) {
                            if (!(ok = warp_wait(bar(L::kOEmpty + 1), oe_ph[1], abort_flag, wf, 20, tile))) break;
                            oe_ph[1] ^= 1;
                        }
                        if (!(ok = warp_wait(bar(L::kPFull + 1), p_ph[1], abort_flag, wf, 22, tile))) break;
                        p_ph[1] ^= 1;
                        tc_fence_after_sync();
                        mma_pv<D, VAR, DV>(tm, sb, 1, vs, j > 0, leader);
                        if constexpr (!kSoftmaxFreesKV) commit(L::kKVEmpty + vs);
                        if (kn >= 0) {
                            mma_qk<D, VAR, DV>(tm, sb, 1, kn, tn, leader);
                            commit(L::kSFull + 1);
                            if constexpr (!kSoftmaxFreesKV) commit(L::kKVEmpty + kn);
                            release_tail(tn);
                            if (j + 2 == nk) commit(L::kQEmpty + 1);
                        } else {
                            commit(L::kOFull + 1);
                            if constexpr (kSoftmaxFreesKV) commit(L::kKVEmpty + vs);  // the work tile's last V
                        }
                    }
                    if (!ok) break;
                }
            }
            // every MMA this warp issued has completed before TMEM is released (with
            // split P the drain counts one commit from each MMA warp)
            if (issued || L::kSplitP) {
                commit(L::kDrain);
                mbar_settle(bar(L::kDrain), 0, wf, 23);
            }
            __syncwarp();
        }
    }
done:
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

}  // namespace fa
