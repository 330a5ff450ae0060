// Attention backward for sm_103a (D = 64 and 128): recompute P from the saved
// log-sum-exp and form the five matrix products of the gradient on the
// tcgen05 tensor cores (FlashAttention from Scratch, sec. 8 "Backward: spend
// arithmetic to save memory"; FlashAttention-4: Blackwell Attention Kernel
// Co-Design, "TMEM backward pipeline").
//
// With c the softmax scale, per (batch, query head):
//   delta_i = O_i . dO_i                       (preprocess kernel)
//   P^T  = 2^(c log2e K Q^T - lse2)            S^T = K Q^T on the tensor core
//   dP^T = V dO^T                              tensor core
//   dV  += P^T dO                              tensor core, P^T from TMEM
//   dS^T = c P^T * (dP^T - delta)              softmax warps, bf16 to shared memory
//   dK  += dS^T Q                              tensor core
//   dQ   = dS K                                tensor core, then TMA reduce-adds to global
//
// Ownership (sec. 8, "A GPU backward must handle competing ownership
// requirements"): a CTA owns one 128-key tile of one KV head and loops over
// every query head of its group and every Q tile that can see the keys, so
// dK and dV are finished in tensor memory without atomics (grouped-query
// heads add into the same accumulators); dQ needs a reduction over key tiles.
// Each step's dQ partial (query rows on the TMEM lanes) is staged in the Q
// stage that dK has just released and added to global memory by TMA fp32
// reduce-adds, which keep the reductions off the SM's memory pipeline.
// Q-tile order is rotated by the key-tile index so that CTAs of the same head
// do not all add into the same dQ rows at the same time.
//
// Tensor memory (512 columns): [0,128) S^T, overwritten by P^T (bf16 pairs);
// [128,256) dP^T, then the dQ partial of the same step; [256,384) dV;
// [384,512) dK.  Shared memory: K and V of the tile; a 3-stage ring of Q
// tiles (each with its lse2 row), because S^T of the next step is issued
// before the current step's dK has released its Q; one dO stage, released by
// P.V halfway through a step; a 2-stage ring of delta rows; and one dS^T tile
// that serves as the K-major A operand of dK and the MN-major A operand of dQ.
//
// Roles (512 threads, one persistent CTA per SM):
//   warps 0-3   thread t owns TMEM lane t: reads query row t of the dQ
//               partial out of TMEM, stages it and sends it with TMA
//               reduce-adds into global dQ; at the end of a work item writes
//               dK and dV (key t)
//   warps 4-11  two groups of four warps, one per half of the 128 query
//               columns; lane t of a group owns key t of the tile.  Each
//               forms its half of P^T (into TMEM, for dV) and of dS^T (into
//               shared memory, for dK and dQ), keeping P^T in registers
//   warp  12    TMA producer      warp 13  MMA issuer, TMEM owner
//   warps 14-15 idle (they complete the last warpgroup for setmaxnreg)
// Registers after setmaxnreg: warps 0-3 192, warps 4-11 128, warps 12-15 64
// (128*192 + 256*128 + 128*64 = 65536, the launch's 128 per thread).
// The dQ reductions (64 KB per step) run on their own warps, overlapped with
// everything else; halving P and dS per thread shortens the chain
// dS -> dK/dQ -> dQ read-out -> dP -> dS that bounds a step.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "fa_bwd.h"
#include "ptx_sm103.cuh"

namespace fa {

// ------------------------------------------------------------------ preprocess

// One warp per (batch * head, row) of the padded row range: delta = O . dO,
// lse2 = LSE * log2(e) (+inf where the row saw no key, so that P = 0), and
// the row of dQ zeroed for the reduce-adds of the main kernel.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdParams p)
{
    constexpr int V = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 8 + warp;  // over B*Hq*Lq_pad
    if (row >= (long long)p.B * p.Hq * p.Lq_pad) return;
    const long long bh = row / p.Lq_pad;
    const int i = (int)(row - bh * p.Lq_pad);
    float delta = 0.f, l2 = INFINITY;
    if (i < p.Lq) {
        const long long r = bh * p.Lq + i;
        const float* o = p.o + r * D + lane * V;
        const uint16_t* g = p.dout + r * D + lane * V;
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < V; ++e) acc = fmaf(o[e], __uint_as_float((uint32_t)g[e] << 16), acc);
#pragma unroll
        for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
        delta = acc;
        const float l = p.lse[r];
        l2 = l == -INFINITY ? INFINITY : l * 1.4426950408889634f;
        float* dq = p.dq + r * D + lane * V;
#pragma unroll
        for (int e = 0; e < V; ++e) dq[e] = 0.f;
    }
    if (lane == 0) {
        p.delta[row] = delta;
        p.lse2[row] = l2;
    }
}

// Largest s in [0, n) with a[s] <= x (a non-decreasing, a[0] <= x).
__device__ __forceinline__ int bwd_upper_index(const int* a, int n, int x)
{
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(a + mid) <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Packed batches, one warp per row, in three ranges of blocks:
//   [0, nb1)        query token rows (token, head): dQ row zeroed;
//   [nb1, nb2)      padded workspace rows (head, padded row): delta and lse2
//                   of the sequence's row, or 0 / +inf on padding rows;
//   [nb2, gridDim)  key token rows (token, KV head) of sequences without
//                   work items (no query rows, or invalid offsets): dK and
//                   dV rows zeroed, since no item writes them.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_varlen_kernel(const BwdParams p, int nb1, int nb2)
{
    constexpr int V = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = p.num_seqs;
    if ((int)blockIdx.x < nb1) {
        const long long row = (long long)blockIdx.x * 8 + warp;  // token * Hq + head
        if (row >= (long long)p.total_q * p.Hq) return;
        float* dq = p.dq + row * D + lane * V;
#pragma unroll
        for (int e = 0; e < V; ++e) dq[e] = 0.f;
    } else if ((int)blockIdx.x < nb2) {
        const long long row = (long long)(blockIdx.x - nb1) * 8 + warp;  // head * Lq_pad + padded row
        if (row >= (long long)p.Hq * p.Lq_pad) return;
        const int h = (int)(row / p.Lq_pad);
        const int r = (int)(row - (long long)h * p.Lq_pad);
        const int* pad = p.sched + 3 * n + 2;
        const int s = bwd_upper_index(pad, n, r);
        const int i = r - __ldg(pad + s);
        const int q0 = __ldg(p.cu_q + s), lq = __ldg(p.cu_q + s + 1) - q0;
        float delta = 0.f, l2 = INFINITY;
        if (r < __ldg(pad + n) && i < lq) {
            const long long t = (long long)(q0 + i) * p.Hq + h;
            const float* o = p.o + t * D + lane * V;
            const uint16_t* g = p.dout + t * D + lane * V;
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < V; ++e) acc = fmaf(o[e], __uint_as_float((uint32_t)g[e] << 16), acc);
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
            delta = acc;
            const float l = p.lse[(long long)h * p.total_q + q0 + i];
            l2 = l == -INFINITY ? INFINITY : l * 1.4426950408889634f;
        }
        if (lane == 0) {
            p.delta[row] = delta;
            p.lse2[row] = l2;
        }
    } else {
        const long long row = (long long)(blockIdx.x - nb2) * 8 + warp;  // key token * Hkv + KV head
        if (row >= (long long)p.total_k * p.Hkv) return;
        const int tok = (int)(row / p.Hkv);
        const int s = bwd_upper_index(p.cu_k, n, tok);
        if (__ldg(p.sched + 2 + 2 * n + s) > 0) return;  // the sequence's items write these rows
        float* dk = p.dk + row * D + lane * V;
        float* dv = p.dv + row * D + lane * V;
#pragma unroll
        for (int e = 0; e < V; ++e) {
            dk[e] = 0.f;
            dv[e] = 0.f;
        }
    }
}

namespace {

constexpr int kBwdThreads = 512;
constexpr int kBox = kBwdTile * 64 * 2;  // one 64-column box of 128 rows (16 KB), a 128-byte swizzle block

// Shared memory and tensor memory of the gradient kernel for head dimension D.
template <int D>
struct BwdSmem {
    static constexpr int kTile = kBwdTile * D * 2;             // one 128-row tile of Q, K, V or dO
    static constexpr int kBoxes = kTile / kBox;                // 64-column boxes per tile
    static constexpr int kDSBytes = kBwdTile * kBwdTile * 2;   // dS^T [128 keys][128 queries] bf16
    // K and V of a work item; at D = 64 in two stages, so that the next
    // item's tiles load while the current item runs
    static constexpr int kKVStages = D == 64 ? 2 : 1;
    static constexpr int kK(int st) { return st * 2 * kTile; }
    static constexpr int kV(int st) { return st * 2 * kTile + kTile; }
    static constexpr int kQStages = 3;
    static constexpr int kQ = kKVStages * 2 * kTile;           // [3] Q tiles
    static constexpr int kDO = kQ + kQStages * kTile;          // dO tile (one stage: free after P.V)
    static constexpr int kDS = kDO + kTile;                    // dS^T
    static constexpr int kL2 = kDS + kDSBytes;                 // [3] lse2 rows (fp32 x 128), with Q
    static constexpr int kDL = kL2 + kQStages * 512;           // [2] delta rows (fp32 x 128)
    static constexpr int kBars = kDL + 2 * 512;
    static constexpr int bKVFull = 0, bKVEmpty = 1, bQFull = 2, bQEmpty = 5, bDOFull = 8, bDOEmpty = 9,
                         bDLFull = 10, bDLEmpty = 12, bSFull = 14, bPFull = 15, bDPFull = 16, bDSFull = 17,
                         bDSEmpty = 18, bDQFull = 19, bDQEmpty = 20, bDKVFull = 21, bDKVEmpty = 22, bDrain = 23,
                         bKV1 = 24, kNumBars = 24 + 2 * (kKVStages - 1);
    static constexpr int bKVFullS(int st) { return st == 0 ? bKVFull : bKV1; }
    static constexpr int bKVEmptyS(int st) { return st == 0 ? bKVEmpty : bKV1 + 1; }
    static constexpr int kMisc = kBars + kNumBars * 8;
    static constexpr int kBytes = kMisc + 16;
    // all the shared memory a CTA may have; the part beyond kBytes absorbs the
    // alignment of the dynamic window to 1024 bytes (checked at run time)
    static constexpr int kDynamic = 232448;
    static_assert(kBytes <= kDynamic, "shared memory of one CTA");
    // Tensor memory columns: S^T (then P^T), dP^T, dV, dK.  dQ (lanes = query
    // rows, D columns) reuses the dP^T columns at D = 128 and has columns of its
    // own at D = 64.
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
    static constexpr uint32_t kColDQ = D == 128 ? kColDP : 256 + 2 * D;
};

constexpr uint32_t kBwdTmemCols = 512;

__device__ __forceinline__ void bwd_tmem_st16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void bwd_fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned, size a multiple of 16),
// completion counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// TMA reduce-add of one 3-D fp32 box from shared memory into global memory
// (a bulk group of the issuing thread), and the waits on such groups.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z)
{
    asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2, %3}], [%4];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

__device__ __forceinline__ float bwd_rcp_approx(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t bwd_pack_bf16(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Three barrier phases tested by back-to-back try_waits of one thread (all
// lanes execute it, so the warp stays converged): the shared-memory round
// trips overlap.  True when all three phases have completed.
__device__ __forceinline__ bool bwd_try_wait3(uint32_t b0, uint32_t p0, uint32_t b1, uint32_t p1, uint32_t b2,
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

__device__ __forceinline__ bool bwd_warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              const WaitFailure& wf, int site, int item)
{
    const bool ok = mbar_wait(bar, parity, abort_flag, wf, site, item);
    return __all_sync(0xffffffffu, ok);
}

// One work item: a 128-key tile of one (batch, KV head); its steps run over
// the query heads of the group (outer) and the Q tiles that can see any key
// of the tile (inner, rotated by the tile index).
struct BwdItem {
    int b, hkv, j;      // batch, KV head, key tile
    int i_min, nq;      // first Q tile with an allowed pair; Q tiles per head
    int i_max;          // last Q tile with an allowed pair
    int steps;          // group * (nq - i_min)
    int lq, lk;         // query / key length of this problem
    int q0, k0;         // packed batches: first query / key token of the sequence
    int ws0;            // packed batches: the sequence's padded workspace row offset
};

// Item r of `slabs` (batch, KV head) slabs of nk key tiles each, in sections
// of hs slabs: section outer, key tile next (longest items first under
// causal), slab innermost.  The items in flight then reduce into the dQ of
// one section's heads only, which stays in L2 between the key tiles.
__device__ __forceinline__ void bwd_section_order(int r, int slabs, int nk, int hs, int& j, int& slab)
{
    const int sec = r / (hs * nk);
    const int rem = r - sec * hs * nk;
    const int cur = min(hs, slabs - sec * hs);
    j = rem / cur;
    slab = sec * hs + (rem - j * cur);
}

template <bool CAUSAL, bool VARLEN, int VAR>
__device__ __forceinline__ BwdItem bwd_item(const BwdParams& p, int it)
{
    BwdItem w;
    if constexpr (VARLEN) {
        // sequences longest query range first; inside one, KV heads in
        // sections, key tiles in order
        const int n = p.num_seqs;
        const int lo = bwd_upper_index(p.sched + 1, n, it);
        const int s = __ldg(p.sched + 2 + n + lo);
        const int rem = it - __ldg(p.sched + 1 + lo);
        w.q0 = __ldg(p.cu_q + s);
        w.lq = __ldg(p.cu_q + s + 1) - w.q0;
        w.k0 = __ldg(p.cu_k + s);
        w.lk = __ldg(p.cu_k + s + 1) - w.k0;
        w.ws0 = __ldg(p.sched + 3 * n + 2 + s);
        bwd_section_order(rem, p.Hkv, (w.lk + kBwdTile - 1) / kBwdTile, p.heads_per_section, w.j, w.hkv);
        w.b = 0;
        w.nq = (w.lq + kBwdTile - 1) / kBwdTile;
    } else {
        int bh;
        bwd_section_order(it, p.B * p.Hkv, p.num_kv_tiles, p.heads_per_section, w.j, bh);
        w.b = bh / p.Hkv;
        w.hkv = bh - w.b * p.Hkv;
        w.nq = p.num_q_tiles;
        w.lq = p.Lq;
        w.lk = p.Lk;
        w.q0 = w.k0 = w.ws0 = 0;
    }
    w.i_min = 0;
    if (CAUSAL) {
        // key k is visible from query q iff k <= q + (Lk - Lq): the tile's first
        // key j*128 needs q >= j*128 - (Lk - Lq)
        const long long first_q = (long long)w.j * kBwdTile - (w.lk - w.lq);
        w.i_min = first_q > 0 ? (int)(first_q / kBwdTile) : 0;
        if (w.i_min > w.nq) w.i_min = w.nq;
    }
    w.i_max = w.nq - 1;
    if (var_window(VAR)) {
        // queries q that see a key of the tile: c_q - left <= key <= c_q + right
        // for some key of [j*128, j*128+127], with c_q = q + (Lk - Lq)
        const long long off = w.lk - w.lq, k0 = (long long)w.j * kBwdTile;
        auto floor_div = [](long long x) { return x >= 0 ? x / kBwdTile : -((-x + kBwdTile - 1) / kBwdTile); };
        long long lo = 0, hi = w.nq - 1;
        if (p.win_right >= 0) lo = max(lo, floor_div(k0 - p.win_right - off));
        if (p.win_left >= 0) hi = min(hi, floor_div(k0 + kBwdTile - 1 + p.win_left - off));
        if (hi < lo) hi = lo = min(lo, (long long)w.nq - 1);  // no pair: one fully masked step gives dK = dV = 0
        w.i_min = (int)lo;
        w.i_max = (int)hi;
    }
    w.steps = p.group * (w.i_max - w.i_min + 1);
    return w;
}

// The k-th work item of this CTA: rounds of gridDim.x items; under causal
// masking (items longest first) the direction alternates from round to round
// so that long and short items pair up on each CTA (balance 0.93 -> 0.997 on
// a causal 16K sequence).
template <bool ALTERNATE>
__device__ __forceinline__ int bwd_cta_item(int k)
{
    const int g = (int)gridDim.x;
    return k * g + ((ALTERNATE && (k & 1)) ? g - 1 - (int)blockIdx.x : (int)blockIdx.x);
}

// Query head and Q tile of step s of an item.
__device__ __forceinline__ void bwd_step(const BwdParams& p, const BwdItem& w, int s, int& h, int& i)
{
    const int span = w.i_max - w.i_min + 1;
    const int g = s / span;
    const int r = s - g * span;
    h = w.hkv * p.group + g;
    i = w.i_min + (r + w.j) % span;
}

}  // namespace

// ------------------------------------------------------------------ main kernel

template <int D, bool CAUSAL, bool VARLEN, int VAR = kVarNone>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_sm103_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                        const __grid_constant__ CUtensorMap tmDQ, const BwdParams p)
{
    using L = BwdSmem<D>;
    constexpr uint32_t kColS = L::kColS, kColDP = L::kColDP, kColDV = L::kColDV, kColDK = L::kColDK,
                       kColDQ = L::kColDQ;
    constexpr int kHalf = kBox;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    auto bar = [&](int i) -> uint32_t { return sb + L::kBars + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WaitFailure wf{p.err, p.diag};
    if ((uint32_t)(smem - smem_raw) + L::kBytes > (uint32_t)L::kDynamic) {
        // the dynamic window is aligned too loosely for the layout: report, touch nothing
        if (threadIdx.x == 0) atomicOr(p.err, 4);
        return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::kKVStages; ++i) {
            mbar_init(bar(L::bKVFullS(i)), 1);
            mbar_init(bar(L::bKVEmptyS(i)), 1);
        }
        for (int i = 0; i < L::kQStages; ++i) {
            mbar_init(bar(L::bQFull + i), 1);
            mbar_init(bar(L::bQEmpty + i), 4);  // each dQ warp, once its staged dQ boxes have been read
        }
        mbar_init(bar(L::bDOFull), 1);
        mbar_init(bar(L::bDOEmpty), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(L::bDLFull + i), 1);
            mbar_init(bar(L::bDLEmpty + i), 256);
        }
        mbar_init(bar(L::bSFull), 1);
        mbar_init(bar(L::bPFull), 256);
        mbar_init(bar(L::bDPFull), 1);
        mbar_init(bar(L::bDSFull), 256);
        mbar_init(bar(L::bDSEmpty), 1);
        mbar_init(bar(L::bDQFull), 1);
        mbar_init(bar(L::bDQEmpty), 128);
        mbar_init(bar(L::bDKVFull), 1);
        mbar_init(bar(L::bDKVEmpty), 128);
        mbar_init(bar(L::bDrain), 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 12 && lane == 0) {
        tma_prefetch_map(&tmQ);
        tma_prefetch_map(&tmK);
        tma_prefetch_map(&tmV);
        tma_prefetch_map(&tmDO);
        tma_prefetch_map(&tmDQ);
    }
    if (warp == 13) {
        tmem_alloc(smem_u32(tmem_slot), kBwdTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int num_items = VARLEN ? __ldg(p.sched) : p.num_items;
    constexpr bool kAlt = CAUSAL || VARLEN || VAR != kVarNone;  // items of unequal length: alternate the rounds

    if (warp < 4) {
        // ============================================================ dQ reduction, dK/dV epilogue
        // Thread t owns TMEM lane t: query row t of the dQ partial (D
        // columns), key t for dK and dV.
        regs_increase<192>();
        const int t = threadIdx.x;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        uint32_t gstep = 0;
        int I = 0;
        for (int k = 0, it = bwd_cta_item<kAlt>(0); it < num_items; it = bwd_cta_item<kAlt>(++k)) {
            const BwdItem w = bwd_item<CAUSAL, VARLEN, VAR>(p, it);
            for (int s = 0; s < w.steps; ++s, ++gstep) {
                int h, i;
                bwd_step(p, w, s, h, i);
                if (!bwd_warp_wait(bar(L::bDQFull), gstep & 1u, abort_flag, wf, 84, it)) goto done;
                tc_fence_after_sync();
                // dK and dQ have completed: their operands dS^T and Q(step) are free.
                // Released here rather than by MMA-warp commits, each of which holds
                // the MMA warp for about 100 cycles with the tensor pipe idle.
                if (t == 0) mbar_arrive(bar(L::bDSEmpty));
                const int q0 = i * kBwdTile;  // dQ rows: dense [B, Hq, Lq, D], packed [Tq, Hq, D]
                if constexpr (D == 128) {
                    uint32_t v0[32], v1[32], v2[32], v3[32];  // query row t: head dimension 0..127
                    tmem_ld32(lane_base + kColDQ, v0);
                    tmem_ld32(lane_base + kColDQ + 32, v1);
                    tmem_ld32(lane_base + kColDQ + 64, v2);
                    tmem_ld32(lane_base + kColDQ + 96, v3);
                    tmem_wait_ld();
                    tc_fence_before_sync();
                    mbar_arrive(bar(L::bDQEmpty));
                    // The partial goes out through this step's Q stage, free now that
                    // dK has read it (the next Q load into it is 1.5 steps away), by
                    // TMA reduce-adds instead of warp-wide red.global.add, which would
                    // hold the SM's memory pipeline for thousands of cycles and delay
                    // the next dS^T stores.  Warp w stages its 32 rows as [32][32] fp32
                    // boxes with the 128-byte swizzle (each thread stores its own row,
                    // 16 bytes at a time, without bank conflicts), two boxes per round.
                    // Rows past Lq are clipped by the tensor map; rows of a packed batch
                    // past the sequence's end hold exact zeros (P = 0 there), which
                    // leave the next sequence's dQ unchanged.
                    const int lane = t & 31;
                    const uint32_t stg = sb + L::kQ + (gstep % L::kQStages) * L::kTile + (uint32_t)(warp * 8192);
                    const int y0 = VARLEN ? h : q0 + 32 * warp;
                    const int z0 = VARLEN ? w.q0 + q0 + 32 * warp : w.b * p.Hq + h;
                    const uint32_t row = stg + (uint32_t)(lane * 128);
#pragma unroll
                    for (int rd = 0; rd < 2; ++rd) {
#pragma unroll
                        for (int bx = 0; bx < 2; ++bx) {
                            const uint32_t* v = rd == 0 ? (bx == 0 ? v0 : v1) : (bx == 0 ? v2 : v3);
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                sts128(row + (uint32_t)(bx * 4096 + ((c ^ (lane & 7)) << 4)), v[4 * c], v[4 * c + 1],
                                       v[4 * c + 2], v[4 * c + 3]);
                        }
                        bwd_fence_proxy_async();
                        __syncwarp();
                        if (lane == 0) {
#pragma unroll
                            for (int bx = 0; bx < 2; ++bx)
                                tma_reduce_add_3d(&tmDQ, stg + (uint32_t)(bx * 4096), 64 * rd + 32 * bx, y0, z0);
                            bulk_commit_group();
                            bulk_wait_read_all();  // the boxes have been read: the stage may be rewritten
                        }
                        __syncwarp();
                    }
                    if (lane == 0) mbar_arrive(bar(L::bQEmpty + (int)(gstep % L::kQStages)));
                } else {
                    uint32_t v0[32], v1[32];  // query row t: head dimension 0..63
                    tmem_ld32(lane_base + kColDQ, v0);
                    tmem_ld32(lane_base + kColDQ + 32, v1);
                    tmem_wait_ld();
                    tc_fence_before_sync();
                    mbar_arrive(bar(L::bDQEmpty));
                    // as at D = 128, through this step's (16 KB) Q stage: one [32][32]
                    // box per warp and round, two rounds
                    const int lane = t & 31;
                    const uint32_t stg = sb + L::kQ + (gstep % L::kQStages) * L::kTile + (uint32_t)(warp * 4096);
                    const int y0 = VARLEN ? h : q0 + 32 * warp;
                    const int z0 = VARLEN ? w.q0 + q0 + 32 * warp : w.b * p.Hq + h;
                    const uint32_t row = stg + (uint32_t)(lane * 128);
#pragma unroll
                    for (int rd = 0; rd < 2; ++rd) {
                        const uint32_t* v = rd == 0 ? v0 : v1;
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            sts128(row + (uint32_t)((c ^ (lane & 7)) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2],
                                   v[4 * c + 3]);
                        bwd_fence_proxy_async();
                        __syncwarp();
                        if (lane == 0) {
                            tma_reduce_add_3d(&tmDQ, stg, 32 * rd, y0, z0);
                            bulk_commit_group();
                            bulk_wait_read_all();
                        }
                        __syncwarp();
                    }
                    if (lane == 0) mbar_arrive(bar(L::bQEmpty + (int)(gstep % L::kQStages)));
                }
            }
            // dK and dV of the finished key tile (thread = key)
            if (!bwd_warp_wait(bar(L::bDKVFull), (uint32_t)(I & 1), abort_flag, wf, 85, it)) goto done;
            tc_fence_after_sync();
            const int key = w.j * kBwdTile + t;
            const long long orow = VARLEN ? (long long)(w.k0 + key) * p.Hkv + w.hkv
                                          : ((long long)w.b * p.Hkv + w.hkv) * p.Lk + key;
#pragma unroll
            for (int o = 0; o < 2; ++o) {
                float* out = (o == 0 ? p.dv : p.dk) + orow * D;
                const uint32_t col = o == 0 ? kColDV : kColDK;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + col + c * 32, r);
                    tmem_wait_ld();
                    if (key < w.lk) {
                        float4* o4 = reinterpret_cast<float4*>(out + c * 32);
#pragma unroll
                        for (int u = 0; u < 8; ++u)
                            o4[u] = make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                                                __uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3]));
                    }
                }
            }
            tc_fence_before_sync();
            mbar_arrive(bar(L::bDKVEmpty));
            ++I;
        }
    } else if (warp < 12) {
        // ============================================================ P^T and dS^T
        // Two groups of four warps, one per half of the Q tile's 128 columns;
        // lane t of a group owns TMEM lane t = key t of the tile.  A thread
        // keeps its half of P^T in registers for dS^T, so the next S^T may
        // overwrite P^T as soon as P.V has read it.
        const int t = 32 * (warp & 3) + lane;
        const int ch = (warp - 4) >> 2;  // column half: queries 64ch .. 64ch+63
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        uint32_t gstep = 0;
        for (int k = 0, it = bwd_cta_item<kAlt>(0); it < num_items; it = bwd_cta_item<kAlt>(++k)) {
            const BwdItem w = bwd_item<CAUSAL, VARLEN, VAR>(p, it);
            const int kpos = w.j * kBwdTile + t;
            const bool key_ok = kpos < w.lk;
            const int off = w.lk - w.lq;
            float alibi_l2 = 0.f;  // ALiBi slope of the step's query head, log2 units
            for (int s = 0; s < w.steps; ++s, ++gstep) {
                int h, i;
                bwd_step(p, w, s, h, i);
                const int q0 = i * kBwdTile;
                const uint32_t ph = gstep & 1u;
                // this step's row statistics: lse2 staged with its Q tile, delta in
                // a ring of its own (both observed here directly, not through the
                // MMA warp)
                const uint32_t qs = gstep % L::kQStages, qph = (gstep / L::kQStages) & 1u;
                const uint32_t ds = gstep & 1u, dph = (gstep >> 1) & 1u;
                const float4* l2p = reinterpret_cast<const float4*>(smem + L::kL2 + qs * 512);
                const float4* dlp = reinterpret_cast<const float4*>(smem + L::kDL + ds * 512);
                // Queries q_lo .. q_hi see this thread's key: q >= key - (Lk - Lq)
                // under the causal mask; with a key window, q >= key - off - right
                // and q <= key - off + left.  A warp masks this step's scores
                // only when one of its keys misses some row of the Q tile.
                constexpr long long kFar = 1ll << 40;  // beyond any token index; no overflow below
                long long q_lo = -kFar, q_hi = kFar;
                if (CAUSAL) q_lo = (long long)kpos - off;
                if constexpr (var_window(VAR)) {
                    if (p.win_right >= 0) q_lo = max(q_lo, (long long)kpos - off - p.win_right);
                    if (p.win_left >= 0) q_hi = (long long)kpos - off + p.win_left;
                }
                if (!key_ok) q_lo = kFar;
                const bool need_mask =
                    __any_sync(0xffffffffu, q_lo > q0 || q_hi < (long long)q0 + kBwdTile - 1);
                if constexpr (var_alibi(VAR)) alibi_l2 = __ldg(p.alibi + h) * 1.4426950408889634f;
                if (!bwd_warp_wait(bar(L::bQFull + qs), qph, abort_flag, wf, 79, it)) goto done;
                if (!bwd_warp_wait(bar(L::bSFull), ph, abort_flag, wf, 80, it)) goto done;
                tc_fence_after_sync();
                // bf16 pairs of queries 64ch + (2e, 2e+1): P, or with soft-capping
                // P * (1 - tanh^2), the factor dS needs
                uint32_t pk[32];
                // the masked and the unmasked step are separate code paths
                auto p_phase = [&](auto masked) {
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = 2 * ch + cc;  // 32-query chunk of the tile
                    // this thread's visible queries as offsets in the chunk, clamped to [-1, 32]
                    const long long cq = (long long)q0 + c * 32;
                    const int e_lo = (int)min(max(q_lo - cq, -1ll), 32ll);
                    const int e_hi = (int)min(max(q_hi - cq, -1ll), 32ll);
                    uint32_t r[32];
                    tmem_ld32(lane_base + kColS + c * 32, r);
                    float l2[32];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float4 v4 = l2p[c * 8 + u];
                        l2[4 * u] = v4.x;
                        l2[4 * u + 1] = v4.y;
                        l2[4 * u + 2] = v4.z;
                        l2[4 * u + 3] = v4.w;
                    }
                    tmem_wait_ld();
                    [[maybe_unused]] uint32_t pt[16];  // soft-capping: this chunk's P for TMEM
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float b0 = -l2[e], b1 = -l2[e + 1];
                        if constexpr (var_alibi(VAR)) {
                            // s' - slope * |c_q - key|, in log2 units (s' = s * scale,
                            // or with soft-capping the capped score below)
                            const float d0 = (float)(q0 + c * 32 + e + off - kpos);
                            b0 = fmaf(-alibi_l2, fabsf(d0), b0);
                            b1 = fmaf(-alibi_l2, fabsf(d0 + 1.f), b1);
                        }
                        float p0, p1;
                        [[maybe_unused]] float g0 = 1.f, g1 = 1.f;  // soft-capping: dt/ds
                        if constexpr (var_softcap(VAR)) {
                            // t = cap tanh(s scale / cap) with tanh(u) = 1 - 2 rho,
                            // rho = 1 / (1 + e^(2u)); dt/ds = 1 - tanh^2 = 4 rho (1 - rho)
                            const float rho0 = bwd_rcp_approx(1.f + ex2_approx(__uint_as_float(r[e]) * p.cap_in2));
                            const float rho1 =
                                bwd_rcp_approx(1.f + ex2_approx(__uint_as_float(r[e + 1]) * p.cap_in2));
                            p0 = ex2_approx(fmaf(fmaf(-2.f, rho0, 1.f), p.cap_out, b0));
                            p1 = ex2_approx(fmaf(fmaf(-2.f, rho1, 1.f), p.cap_out, b1));
                            g0 = 4.f * rho0 * (1.f - rho0);
                            g1 = 4.f * rho1 * (1.f - rho1);
                        } else {
                            p0 = ex2_approx(fmaf(__uint_as_float(r[e]), p.scale_log2, b0));
                            p1 = ex2_approx(fmaf(__uint_as_float(r[e + 1]), p.scale_log2, b1));
                        }
                        if constexpr (decltype(masked)::value) {
                            if (e < e_lo || e > e_hi) p0 = 0.f;
                            if (e + 1 < e_lo || e + 1 > e_hi) p1 = 0.f;
                        }
                        if constexpr (var_softcap(VAR)) {
                            pt[e / 2] = bwd_pack_bf16(p0, p1);
                            pk[cc * 16 + e / 2] = bwd_pack_bf16(p0 * g0, p1 * g1);
                        } else {
                            pk[cc * 16 + e / 2] = bwd_pack_bf16(p0, p1);
                        }
                    }
                    // P^T of this half goes to the first 32 of its own 64 S^T
                    // columns (column 64ch + c holds queries 64ch + 2c, 2c + 1), which
                    // this thread has read; the other half's columns may still be
                    // being read by its warps
                    if constexpr (var_softcap(VAR)) bwd_tmem_st16(lane_base + kColS + 64 * ch + 16 * cc, pt);
                }
                };
                if (need_mask)
                    p_phase(std::true_type{});
                else
                    p_phase(std::false_type{});
                if constexpr (!var_softcap(VAR)) {
                    uint32_t lo[16], hi[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        lo[e] = pk[e];
                        hi[e] = pk[16 + e];
                    }
                    bwd_tmem_st16(lane_base + kColS + 64 * ch, lo);
                    bwd_tmem_st16(lane_base + kColS + 64 * ch + 16, hi);
                }
                tmem_wait_st();
                tc_fence_before_sync();
                mbar_arrive(bar(L::bPFull));
                // dS^T = c P^T (dP^T - delta) for the half's 64 queries
                if (!bwd_warp_wait(bar(L::bDLFull + ds), dph, abort_flag, wf, 77, it)) goto done;
                if (!bwd_warp_wait(bar(L::bDPFull), ph, abort_flag, wf, 82, it)) goto done;
                if (!bwd_warp_wait(bar(L::bDSEmpty), ph ^ 1u, abort_flag, wf, 83, it)) goto done;
                tc_fence_after_sync();
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const int c = 2 * ch + cc;
                    uint32_t r[32];
                    tmem_ld32(lane_base + kColDP + c * 32, r);
                    float dl[32];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const float4 v4 = dlp[c * 8 + u];
                        dl[4 * u] = v4.x;
                        dl[4 * u + 1] = v4.y;
                        dl[4 * u + 2] = v4.z;
                        dl[4 * u + 3] = v4.w;
                    }
                    tmem_wait_ld();
                    uint32_t d[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const uint32_t w2 = pk[cc * 16 + e / 2];
                        const float p0 = __uint_as_float(w2 << 16), p1 = __uint_as_float(w2 & 0xffff0000u);
                        const float ds0 = (__uint_as_float(r[e]) - dl[e]) * (p0 * p.scale);
                        const float ds1 = (__uint_as_float(r[e + 1]) - dl[e + 1]) * (p1 * p.scale);
                        d[e / 2] = bwd_pack_bf16(ds0, ds1);
                    }
                    // dS^T row t, queries 32c .. 32c+31: half ch, 16-byte chunks 4(c&1) .. +3
                    // (the A operand of dQ, read MN-major)
                    const uint32_t row = sb + L::kDS + (uint32_t)(ch * kHalf + t * 128);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int chunk = (c & 1) * 4 + u;
                        sts128(row + (uint32_t)((chunk ^ (t & 7)) << 4), d[4 * u], d[4 * u + 1], d[4 * u + 2],
                               d[4 * u + 3]);
                    }
                    // and in tensor memory as the A operand of dK, laid out like P^T:
                    // the first 32 of this half's 64 dP^T columns, already read
                    bwd_tmem_st16(lane_base + kColDP + 64 * ch + 16 * cc, d);
                }
                tmem_wait_st();
                bwd_fence_proxy_async();
                tc_fence_before_sync();
                mbar_arrive(bar(L::bDSFull));
                mbar_arrive(bar(L::bDLEmpty + ds));
            }
        }
    } else if (warp == 12) {
        // ============================================================ TMA producer
        regs_decrease<64>();
        if (lane == 0) {
            int q_armed[L::kQStages] = {-1, -1, -1}, dl_armed[2] = {-1, -1}, do_armed = -1, kv_armed[2] = {-1, -1};
            bool drop = p.fault == 1;  // test hook: this CTA's first K/V never arrives
            uint32_t gstep = 0;
            int I = 0;
            for (int k = 0, it = bwd_cta_item<kAlt>(0); it < num_items; it = bwd_cta_item<kAlt>(++k)) {
                const BwdItem w = bwd_item<CAUSAL, VARLEN, VAR>(p, it);
                const int bh_kv = w.b * p.Hkv + w.hkv;
                const int st = I % L::kKVStages;
                const uint32_t kvph = (uint32_t)((I / L::kKVStages) & 1);
                // TMA coordinates: dense (x, row, head slab), packed (x, head, token)
                auto ld_kv = [&](uint32_t dst, const CUtensorMap* map, int x) {
                    if constexpr (VARLEN)
                        tma_load_3d(dst, map, bar(L::bKVFullS(st)), x, w.hkv, w.k0 + w.j * kBwdTile);
                    else
                        tma_load_3d(dst, map, bar(L::bKVFullS(st)), x, w.j * kBwdTile, bh_kv);
                };
                if (!mbar_wait(bar(L::bKVEmptyS(st)), kvph ^ 1u, abort_flag, wf, 85, it)) break;
                if (drop) {
                    drop = false;
                } else {
                    mbar_arrive_expect_tx(bar(L::bKVFullS(st)), 2 * L::kTile);
                    kv_armed[st] = (int)kvph;
#pragma unroll
                    for (int bx = 0; bx < L::kBoxes; ++bx) {
                        ld_kv(sb + L::kK(st) + bx * kBox, &tmK, 64 * bx);
                        ld_kv(sb + L::kV(st) + bx * kBox, &tmV, 64 * bx);
                    }
                }
                bool ok = true;
                for (int s = 0; s < w.steps; ++s, ++gstep) {
                    int h, i;
                    bwd_step(p, w, s, h, i);
                    const int y = i * kBwdTile, z = w.b * p.Hq + h;
                    const long long ws_row = VARLEN ? (long long)h * p.Lq_pad + w.ws0 + y : (long long)z * p.Lq_pad + y;
                    // Q/dO coordinates: dense (x, row, head slab), packed (x, head, token)
                    const int c1 = VARLEN ? h : y, c2 = VARLEN ? w.q0 + y : z;
                    // Q and its lse2 row (3-stage ring: freed after dK)
                    const uint32_t qs = gstep % L::kQStages, qph = (gstep / L::kQStages) & 1u;
                    if (!(ok = mbar_wait(bar(L::bQEmpty + qs), qph ^ 1u, abort_flag, wf, 86, it))) break;
                    mbar_arrive_expect_tx(bar(L::bQFull + qs), L::kTile + 512);
                    q_armed[qs] = (int)qph;
                    const uint32_t qdst = sb + L::kQ + qs * L::kTile;
#pragma unroll
                    for (int bx = 0; bx < L::kBoxes; ++bx)
                        tma_load_3d(qdst + bx * kBox, &tmQ, bar(L::bQFull + qs), 64 * bx, c1, c2);
                    bulk_load(sb + L::kL2 + qs * 512, p.lse2 + ws_row, 512, bar(L::bQFull + qs));
                    // delta row (2-stage ring: freed by the dS warps)
                    const uint32_t ds = gstep & 1u, dph = (gstep >> 1) & 1u;
                    if (!(ok = mbar_wait(bar(L::bDLEmpty + ds), dph ^ 1u, abort_flag, wf, 87, it))) break;
                    mbar_arrive_expect_tx(bar(L::bDLFull + ds), 512);
                    dl_armed[ds] = (int)dph;
                    bulk_load(sb + L::kDL + ds * 512, p.delta + ws_row, 512, bar(L::bDLFull + ds));
                    // dO (one stage: freed after P.V)
                    if (!(ok = mbar_wait(bar(L::bDOEmpty), (gstep & 1u) ^ 1u, abort_flag, wf, 88, it))) break;
                    mbar_arrive_expect_tx(bar(L::bDOFull), L::kTile);
                    do_armed = (int)(gstep & 1u);
#pragma unroll
                    for (int bx = 0; bx < L::kBoxes; ++bx)
                        tma_load_3d(sb + L::kDO + bx * kBox, &tmDO, bar(L::bDOFull), 64 * bx, c1, c2);
                }
                if (!ok) break;
                ++I;
            }
            // every copy this thread started has landed before the CTA retires
            for (int st = 0; st < L::kKVStages; ++st)
                if (kv_armed[st] >= 0) mbar_settle(bar(L::bKVFullS(st)), (uint32_t)kv_armed[st], wf, 97);
            for (int t = 0; t < L::kQStages; ++t)
                if (q_armed[t] >= 0) mbar_settle(bar(L::bQFull + t), (uint32_t)q_armed[t], wf, 98);
            for (int t = 0; t < 2; ++t)
                if (dl_armed[t] >= 0) mbar_settle(bar(L::bDLFull + t), (uint32_t)dl_armed[t], wf, 99);
            if (do_armed >= 0) mbar_settle(bar(L::bDOFull), (uint32_t)do_armed, wf, 100);
        }
        __syncwarp();
    } else if (warp == 13) {
        // ============================================================ MMA issuer (warp 13)
        regs_decrease<64>();
        const bool leader = lane == 0;
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        constexpr int kKD = D / 16;                                      // MMAs over the head dimension
        constexpr uint32_t kIdSS = idesc_bf16_f32(128, 128, false);     // S^T, dP^T: A, B K-major
        constexpr uint32_t kIdBmn = idesc_bf16_f32(128, D, true);       // dV, dK: B MN-major, N = D
        // dQ (M = queries, N = head dimension); A and B MN-major
        constexpr uint32_t kIdDQ = idesc_bf16_f32(128, D, true) | (1u << 15);
        auto commit = [&](int b) {
            if (leader) tc_commit(bar(b));
            __syncwarp();
        };
        auto kmaj = [](int kk) -> uint64_t { return (uint64_t)(((kk >> 2) * kHalf + (kk & 3) * 32) >> 4); };
        auto mnmaj = [](int kk) -> uint64_t { return (uint64_t)((kk * 16 * 128) >> 4); };
        // K and V of the current item (stage set per item)
        uint64_t dK_kmaj = 0, dK_mn = 0, dV_kmaj = 0;
        const uint64_t dS_mn = smem_desc_sw128(sb + L::kDS, kHalf, 1024);
        // S^T = K Q^T into the S region
        const uint64_t dO_kmaj = smem_desc_sw128(sb + L::kDO, 16, 1024);
        const uint64_t dO_mn = smem_desc_sw128(sb + L::kDO, kHalf, 1024);
        auto mma_s = [&](uint32_t qs) {
            const uint64_t qd = smem_desc_sw128(sb + L::kQ + qs * L::kTile, 16, 1024);
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kKD; ++kk)
                    mma_ss(tm + kColS, dK_kmaj + kmaj(kk), qd + kmaj(kk), kIdSS, kk > 0);
            }
            __syncwarp();
        };
        uint32_t gstep = 0;
        int I = 0;
        bool issued = false, ok = true;
        for (int k = 0, it = bwd_cta_item<kAlt>(0); it < num_items && ok; it = bwd_cta_item<kAlt>(++k)) {
            const BwdItem w = bwd_item<CAUSAL, VARLEN, VAR>(p, it);
            const int st = I % L::kKVStages;
            if (!(ok = bwd_warp_wait(bar(L::bKVFullS(st)), (uint32_t)((I / L::kKVStages) & 1), abort_flag, wf, 89,
                                     it)))
                break;
            dK_kmaj = smem_desc_sw128(sb + L::kK(st), 16, 1024);
            dK_mn = smem_desc_sw128(sb + L::kK(st), kHalf, 1024);
            dV_kmaj = smem_desc_sw128(sb + L::kV(st), 16, 1024);
            {
                const uint32_t qs = gstep % L::kQStages, qph = (gstep / L::kQStages) & 1u;
                if (!(ok = bwd_warp_wait(bar(L::bQFull + qs), qph, abort_flag, wf, 90, it))) break;
                tc_fence_after_sync();
                mma_s(qs);
                issued = true;
                commit(L::bSFull);
            }
            for (int s = 0; s < w.steps; ++s, ++gstep) {
                const uint32_t qs = gstep % L::kQStages;
                const uint64_t q_mn = smem_desc_sw128(sb + L::kQ + qs * L::kTile, kHalf, 1024);
                // dP^T = V dO^T.  At D = 128 its columns held the previous step's dQ,
                // so it waits for the dQ read-out; at D = 64 dQ has columns of its own
                // and only the dQ MMAs below wait for it, which takes the read-out
                // off the step's chain.  The waits of the MMA warp are tested
                // together first (one shared-memory round trip when, as usual, the
                // phases have completed), then one by one.
                constexpr bool kDQOwnCols = kColDQ != kColDP;
                const bool ready1 = __all_sync(
                    0xffffffffu, bwd_try_wait3(kDQOwnCols ? bar(L::bDOFull) : bar(L::bDQEmpty),
                                               kDQOwnCols ? (gstep & 1u) : ((gstep & 1u) ^ 1u), bar(L::bDOFull),
                                               gstep & 1u, bar(L::bDOFull), gstep & 1u));
                if (!ready1) {
                    if (!kDQOwnCols &&
                        !(ok = bwd_warp_wait(bar(L::bDQEmpty), (gstep & 1u) ^ 1u, abort_flag, wf, 91, it)))
                        break;
                    if (!(ok = bwd_warp_wait(bar(L::bDOFull), gstep & 1u, abort_flag, wf, 101, it))) break;
                }
                tc_fence_after_sync();
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < kKD; ++kk)
                        mma_ss(tm + kColDP, dV_kmaj + kmaj(kk), dO_kmaj + kmaj(kk), kIdSS, kk > 0);
                }
                __syncwarp();
                commit(L::bDPFull);
                // dV += P^T dO (P^T; at an item's first step the dK/dV accumulators;
                // and the next step's Q, tested with them)
                const bool has_next = s + 1 < w.steps;
                const uint32_t q1 = (gstep + 1) % L::kQStages, ph1 = ((gstep + 1) / L::kQStages) & 1u;
                const uint32_t bp = bar(L::bPFull), pp = gstep & 1u;
                const bool ready2 = __all_sync(
                    0xffffffffu,
                    bwd_try_wait3(bp, pp, s == 0 ? bar(L::bDKVEmpty) : bp, s == 0 ? ((uint32_t)(I & 1) ^ 1u) : pp,
                                  has_next ? bar(L::bQFull + q1) : bp, has_next ? ph1 : pp));
                if (!ready2) {
                    if (!(ok = bwd_warp_wait(bp, pp, abort_flag, wf, 92, it))) break;
                    if (s == 0 &&
                        !(ok = bwd_warp_wait(bar(L::bDKVEmpty), (uint32_t)(I & 1) ^ 1u, abort_flag, wf, 93, it)))
                        break;
                }
                tc_fence_after_sync();
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tm + kColDV, tm + kColS + (uint32_t)(kk * 8 + (kk >= 4 ? 32 : 0)), dO_mn + mnmaj(kk),
                               kIdBmn,
                               (s > 0 || kk > 0) ? 1u : 0u);
                }
                __syncwarp();
                commit(L::bDOEmpty);  // dO's last reader
                // next step's S^T: P^T of this step has been consumed (MMAs run in order)
                if (has_next) {
                    if (!ready2) {
                        if (!(ok = bwd_warp_wait(bar(L::bQFull + q1), ph1, abort_flag, wf, 90, it))) break;
                        tc_fence_after_sync();
                    }
                    mma_s(q1);
                    commit(L::bSFull);
                }
                // dK += dS^T Q and dQ = dS K
                if (!(ok = bwd_warp_wait(bar(L::bDSFull), gstep & 1u, abort_flag, wf, 94, it))) break;
                tc_fence_after_sync();
                // dK += dS^T Q with A = dS^T from tensor memory (the P/dS warps' copy
                // in the dP^T columns), which saves its shared-memory reads; dQ = dS K
                // with the query rows on the TMEM lanes (A = dS and B = K both
                // MN-major), so that each dQ thread holds one row
                auto mma_dk = [&] {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tm + kColDK, tm + kColDP + (uint32_t)(kk * 8 + (kk >= 4 ? 32 : 0)), q_mn + mnmaj(kk),
                               kIdBmn, (s > 0 || kk > 0) ? 1u : 0u);
                };
                auto mma_dq = [&] {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tm + kColDQ, dS_mn + mnmaj(kk), dK_mn + mnmaj(kk), kIdDQ, kk > 0);
                };
                if constexpr (kDQOwnCols) {
                    if (leader) mma_dk();
                    __syncwarp();
                    // the previous dQ must have left its columns
                    if (!(ok = bwd_warp_wait(bar(L::bDQEmpty), (gstep & 1u) ^ 1u, abort_flag, wf, 91, it))) break;
                    if (leader) mma_dq();
                } else {
                    if (leader) {
                        mma_dk();
                        mma_dq();
                    }
                }
                __syncwarp();
                commit(L::bDQFull);  // the dQ warps then free dS^T and Q (stage qs)
            }
            if (!ok) break;
            commit(L::bDKVFull);
            commit(L::bKVEmptyS(st));
            ++I;
        }
        if (issued) {
            commit(L::bDrain);
            mbar_settle(bar(L::bDrain), 0, wf, 95);
        }
        __syncwarp();
    } else {
        regs_decrease<64>();  // warps 14-15 only complete the last warpgroup
    }
done:
    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 13) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kBwdTmemCols);
    }
}

#if !defined(FA_BWD_VARIANTS)
cudaError_t launch_bwd_pre(int D, bool varlen, const BwdParams& p, cudaStream_t stream)
{
    if (varlen) {
        const long long r1 = (long long)p.total_q * p.Hq, r2 = (long long)p.Hq * p.Lq_pad,
                        r3 = (long long)p.total_k * p.Hkv;
        const long long nb1 = (r1 + 7) / 8, nb2 = nb1 + (r2 + 7) / 8, nb = nb2 + (r3 + 7) / 8;
        if (nb >= (1ll << 31)) return cudaErrorInvalidValue;
        if (D == 128)
            fa_bwd_pre_varlen_kernel<128><<<(int)nb, 256, 0, stream>>>(p, (int)nb1, (int)nb2);
        else
            fa_bwd_pre_varlen_kernel<64><<<(int)nb, 256, 0, stream>>>(p, (int)nb1, (int)nb2);
        return cudaGetLastError();
    }
    const long long rows = (long long)p.B * p.Hq * p.Lq_pad;
    const int grid = (int)((rows + 7) / 8);
    if (D == 128)
        fa_bwd_pre_kernel<128><<<grid, 256, 0, stream>>>(p);
    else
        fa_bwd_pre_kernel<64><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}
#endif

namespace {
template <int D, bool CAUSAL, bool VARLEN, int VAR = kVarNone>
cudaError_t launch_bwd_kernel(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                              const CUtensorMap& dout, const CUtensorMap& dq, const BwdParams& p, int grid,
                              cudaStream_t stream)
{
    auto kern = fa_bwd_sm103_kernel<D, CAUSAL, VARLEN, VAR>;
    constexpr int kSmem = BwdSmem<D>::kDynamic;
    const cudaError_t e = smem_limit_once<fa_bwd_sm103_kernel<D, CAUSAL, VARLEN, VAR>>(kSmem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kBwdThreads, kSmem, stream>>>(q, k, v, dout, dq, p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_dim(bool causal, bool varlen, const CUtensorMap& q, const CUtensorMap& k,
                           const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& dq, const BwdParams& p,
                           int grid, cudaStream_t stream)
{
    if (varlen)
        return causal ? launch_bwd_kernel<D, true, true>(q, k, v, dout, dq, p, grid, stream)
                      : launch_bwd_kernel<D, false, true>(q, k, v, dout, dq, p, grid, stream);
    return causal ? launch_bwd_kernel<D, true, false>(q, k, v, dout, dq, p, grid, stream)
                  : launch_bwd_kernel<D, false, false>(q, k, v, dout, dq, p, grid, stream);
}
}  // namespace

#if !defined(FA_BWD_VARIANTS)
cudaError_t launch_bwd(int D, bool causal, bool varlen, const CUtensorMap& q, const CUtensorMap& k,
                       const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& dq, const BwdParams& p,
                       int grid, cudaStream_t stream)
{
    if (D == 128) return launch_bwd_dim<128>(causal, varlen, q, k, v, dout, dq, p, grid, stream);
    if (D == 64) return launch_bwd_dim<64>(causal, varlen, q, k, v, dout, dq, p, grid, stream);
    return cudaErrorInvalidValue;
}
#else
#ifndef FA_BWD_HEAD_DIM
#define FA_BWD_HEAD_DIM 128
#endif
#if FA_BWD_HEAD_DIM == 64
#define FA_BWD_VARIANT_FN launch_bwd_variant_d64
#else
#define FA_BWD_VARIANT_FN launch_bwd_variant_d128
#endif
cudaError_t FA_BWD_VARIANT_FN(int var, bool varlen, const CUtensorMap& q, const CUtensorMap& k,
                              const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& dq,
                              const BwdParams& p, int grid, cudaStream_t stream)
{
    constexpr int D = FA_BWD_HEAD_DIM;
    if (var == kVarAlibi)
        return varlen ? launch_bwd_kernel<D, false, true, kVarAlibi>(q, k, v, dout, dq, p, grid, stream)
                      : launch_bwd_kernel<D, false, false, kVarAlibi>(q, k, v, dout, dq, p, grid, stream);
    if (var == kVarWindow)
        return varlen ? launch_bwd_kernel<D, false, true, kVarWindow>(q, k, v, dout, dq, p, grid, stream)
                      : launch_bwd_kernel<D, false, false, kVarWindow>(q, k, v, dout, dq, p, grid, stream);
    if (var == kVarSoftcap)
        return varlen ? launch_bwd_kernel<D, false, true, kVarSoftcap>(q, k, v, dout, dq, p, grid, stream)
                      : launch_bwd_kernel<D, false, false, kVarSoftcap>(q, k, v, dout, dq, p, grid, stream);
    if (var == kVarCapAlibi)
        return varlen ? launch_bwd_kernel<D, false, true, kVarCapAlibi>(q, k, v, dout, dq, p, grid, stream)
                      : launch_bwd_kernel<D, false, false, kVarCapAlibi>(q, k, v, dout, dq, p, grid, stream);
    return cudaErrorInvalidValue;
}
#endif

}  // namespace fa
