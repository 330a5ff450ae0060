// C ABI of the attention library: argument validation, tensor-map encoding,
// scheduling and launch.  Declarations and contracts: include/fa_gb300.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fa_gb300.h"
#include "fa_bwd.h"
#include "fa_decode.h"
#include "fa_fp8.h"
#include "fa_launch.h"
#include "fa_params.h"

namespace fa {

// Device-side error latch: bit 0 = a pipeline wait timed out, bit 1 = invalid
// variable-length offsets, bit 2 = a kernel found its launch configuration
// unusable (shared-memory window alignment) and did nothing.  g_diag keeps the first failing wait site.
__device__ int g_err;
__device__ int g_diag[4];

namespace {

constexpr int kMaxDevices = 64;
// K/V bytes per scheduling section of KV heads.  Work tiles of unequal
// length (causal, key windows, packed batches) need the whole-L2 section so
// that the longest-first order can balance them; equal tiles measured faster
// with sections a quarter of the L2, whose K/V stays in it (fewer re-reads
// from HBM).
constexpr long long kL2SectionBytes = 128ll << 20;
constexpr long long kL2SectionBytesEqualTiles = 32ll << 20;

struct DeviceState {
    bool ready = false;
    fa_status_t status = FA_OK;
    int num_sms = 0;
    int* err = nullptr;
    int* diag = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
thread_local int g_last_launches = 0;
thread_local int g_fault_next = 0;  // test hook, consumed by the next fa_fwd

fa_status_t device_state(DeviceState** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& s = g_dev[dev];
    if (!s.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FA_ERR_CUDA;
        if (major != 10 || minor != 3) {
            s.status = FA_ERR_UNSUPPORTED;  // kernels are built for sm_103a only
        } else {
            if (cudaGetSymbolAddress(reinterpret_cast<void**>(&s.err), g_err) != cudaSuccess ||
                cudaGetSymbolAddress(reinterpret_cast<void**>(&s.diag), g_diag) != cudaSuccess)
                return FA_ERR_CUDA;
            if (!g_encode) {
                cudaDriverEntryPointQueryResult q;
                void* fn = nullptr;
                if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                                     &q) != cudaSuccess ||
                    q != cudaDriverEntryPointSuccess || !fn)
                    return FA_ERR_CUDA;
                g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
            }
        }
        s.ready = true;
    }
    *out = &s;
    return s.status;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D bf16 tensor map with 128-byte swizzle: box = {64, box1, box2} elements.
bool encode_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box1, uint32_t box2)
{
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {64, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D fp32 tensor map with 128-byte swizzle (box0 = 32 elements = one
// swizzle row): box = {box0, box1, box2} elements (the backward's dQ
// reduce-adds).
bool encode_map_f32(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1, uint32_t box2)
{
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {box0, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Dense batches: the (batch, head) slabs of Q, K, V, O and LSE are contiguous,
// so B batches of Hq query heads over Hkv KV heads are one batch of B*Hq query
// heads over B*Hkv KV heads (query head b*Hq + h reads KV head
// (b*Hq + h) / (Hq/Hkv) = b*Hkv + h/(Hq/Hkv)), and the kernel's longest-first
// tile order then spans the whole batch instead of restarting at each batch
// (a causal B = 2 list was 12 % out of balance over 152 CTAs).  ALiBi keeps the
// batch: its slopes are indexed by the query head within the batch.
void set_batch_heads(FwdParams* p, int B, int Hq, int Hkv, bool fold)
{
    p->B = fold ? 1 : B;
    p->Hq = fold ? B * Hq : Hq;
    p->Hkv = fold ? B * Hkv : Hkv;
}

// KV slabs per scheduling section.  slabs = the KV heads of one batch (all
// (batch, KV head) slabs when the batch is folded into the heads) or of one
// packed sequence; D_kv = the K and V bytes of one key / 2 (D + Dv for bf16).
int heads_per_section(int slabs, long long Lk, int D_kv, bool equal_tiles)
{
    const long long kv_bytes = Lk * D_kv * 2;  // K and V of one slab
    const long long budget = equal_tiles ? kL2SectionBytesEqualTiles : kL2SectionBytes;
    long long hs = kv_bytes > 0 ? budget / kv_bytes : slabs;
    if (hs < 1) hs = 1;
    if (hs > slabs) hs = slabs;
    return (int)hs;
}

template <int D, bool VARLEN>
cudaError_t dispatch_variant_dim(int var, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const FwdParams& p, int grid, cudaStream_t st)
{
    if (var == kVarSoftcap) return launch_fwd<D, false, VARLEN, kVarSoftcap>(q, k, v, p, grid, st);
    if (var == kVarAlibi) return launch_fwd<D, false, VARLEN, kVarAlibi>(q, k, v, p, grid, st);
    if (var == kVarCapAlibi) return launch_fwd<D, false, VARLEN, kVarCapAlibi>(q, k, v, p, grid, st);
    return launch_fwd<D, false, VARLEN, kVarWindow>(q, k, v, p, grid, st);
}

// D = 64 or 128 (checked by prepare_variant)
template <bool VARLEN>
cudaError_t dispatch_variant(int D, int var, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const FwdParams& p, int grid, cudaStream_t st)
{
    return D == 64 ? dispatch_variant_dim<64, VARLEN>(var, q, k, v, p, grid, st)
                   : dispatch_variant_dim<128, VARLEN>(var, q, k, v, p, grid, st);
}

// Validates a variant description and fills the kernel parameters; returns
// the variant kind (kVar*) or a negative fa_status_t.
int prepare_variant(const fa_variant_t* var, int D, float scale, FwdParams* p)
{
    if (!var) return -(int)FA_ERR_INVALID_ARG;
    if (!std::isfinite(var->softcap) || var->softcap < 0.f) return -(int)FA_ERR_INVALID_ARG;
    if (var->alibi_slopes && (reinterpret_cast<uintptr_t>(var->alibi_slopes) & 3u)) return -(int)FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return -(int)FA_ERR_UNSUPPORTED;
    p->win_left = var->window_left < 0 ? -1 : var->window_left;
    p->win_right = var->window_right < 0 ? -1 : var->window_right;
    p->alibi = var->alibi_slopes;
    if (var->softcap > 0.f) {
        p->cap_in = scale / var->softcap;
        p->cap_out = (float)((double)var->softcap * 1.4426950408889634);
        return var->alibi_slopes ? kVarCapAlibi : kVarSoftcap;
    }
    return var->alibi_slopes ? kVarAlibi : kVarWindow;
}

// Key windows: whether the last 256-row block of an Lq x Lk problem sees at
// least as many KV tiles as the first (a causal-like window), in which case
// the kernel takes row blocks from the last, longest first (the same window
// arithmetic as the kernel's tile decoding).
int window_tiles_desc(const FwdParams& p, long long Lq, long long Lk)
{
    if (Lq <= 0 || Lk <= 0) return 0;
    auto kv_tiles = [&](long long m0) -> long long {
        const long long off = Lk - Lq, last_row = std::min(m0 + kRowsPerCta - 1, Lq - 1);
        const long long lo = p.win_left >= 0 ? std::max(0ll, m0 + off - p.win_left) : 0;
        const long long hi = p.win_right >= 0 ? std::min(Lk - 1, last_row + off + p.win_right) : Lk - 1;
        return hi < lo ? 0 : hi / kBlockN - lo / kBlockN + 1;
    };
    const long long last_m0 = (Lq - 1) / kRowsPerCta * kRowsPerCta;
    return kv_tiles(last_m0) >= kv_tiles(0) ? 1 : 0;
}

// (D, Dv) must satisfy hdim_supported()
template <bool VARLEN>
cudaError_t dispatch(int D, bool causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                     const FwdParams& p, int grid, cudaStream_t st)
{
    if (D == 192)
        return causal ? launch_fwd<192, true, VARLEN, kVarNone, 128>(q, k, v, p, grid, st)
                      : launch_fwd<192, false, VARLEN, kVarNone, 128>(q, k, v, p, grid, st);
    if (D == 64)
        return causal ? launch_fwd<64, true, VARLEN>(q, k, v, p, grid, st)
                      : launch_fwd<64, false, VARLEN>(q, k, v, p, grid, st);
    return causal ? launch_fwd<128, true, VARLEN>(q, k, v, p, grid, st)
                  : launch_fwd<128, false, VARLEN>(q, k, v, p, grid, st);
}

bool scale_ok(float s) { return std::isfinite(s) && s > 0.f; }

// Head dimensions with a kernel: (64, 64), (128, 128) and (192, 128).
bool hdim_supported(int D, int Dv) { return (D == Dv && (D == 64 || D == 128)) || (D == 192 && Dv == 128); }

}  // namespace

// --------------------------------------------------------------- varlen schedule

// One CTA of 1024 threads.  Validates the offsets, orders sequences by the
// length of their longest work tile, longest first (FlashAttention-4:
// Blackwell Attention Kernel Co-Design, "LPT scheduling for imbalanced
// grids", step 4), and writes the exclusive prefix of work tiles in that
// order.
//   forward  (bwd = 0): a tile is 256 query rows of one query head and visits
//            ceil(Lk/128) KV tiles: tiles = Hq * ceil(Lq/256), sorted by Lk;
//            with paired heads (bwd = 2) 128 rows of two query heads:
//            tiles = (Hq/2) * ceil(Lq/128).
//   backward (bwd = 1): an item is 128 keys of one KV head and visits the Q
//            tiles of the group: items = Hkv * ceil(Lk/128) when Lq > 0,
//            sorted by Lq; also the sequences' row offsets in a workspace
//            where each sequence's rows are padded to a multiple of 128.
//
// sched layout (int32): [0] total tiles | [1 .. n+1] prefix by schedule rank |
// [n+2 .. 2n+1] order (rank -> sequence) | [2n+2 .. 3n+1] tiles by sequence |
// backward only: [3n+2 .. 4n+2] padded row offset of each sequence (original
// order, n+1 entries).
constexpr int kSchedThreads = 1024;
constexpr int kSortMax = 4096;

__global__ void __launch_bounds__(kSchedThreads)
    fa_varlen_schedule_kernel(const int* __restrict__ cu_q, const int* __restrict__ cu_k, int n, int total_q,
                              int total_k, int max_q, int max_k, int heads, int bwd, int* __restrict__ sched,
                              int* __restrict__ err)
{
    __shared__ int key[kSortMax];
    __shared__ int part[kSchedThreads];
    __shared__ int bad;
    const int tid = threadIdx.x;
    int* prefix = sched + 1;
    int* order = sched + 2 + n;
    int* tiles = sched + 2 + 2 * n;
    if (tid == 0) bad = (cu_q[0] != 0 || cu_k[0] != 0 || cu_q[n] != total_q || cu_k[n] != total_k) ? 1 : 0;
    __syncthreads();
    // per-sequence check; an invalid sequence is scheduled with no work
    for (int s = tid; s < n; s += kSchedThreads) {
        const int q0 = cu_q[s], q1 = cu_q[s + 1], k0 = cu_k[s], k1 = cu_k[s + 1];
        const bool ok = !bad && q0 >= 0 && q1 >= q0 && q1 <= total_q && q1 - q0 <= max_q && k0 >= 0 &&
                        k1 >= k0 && k1 <= total_k && k1 - k0 <= max_k;
        if (!ok) atomicOr(err, 2);
        if (bwd == 1) {
            if (n <= kSortMax) key[s] = (ok && q1 > q0 && k1 > k0) ? (q1 - q0) : -1;
            tiles[s] = (ok && q1 > q0) ? heads * ((k1 - k0 + 127) / 128) : 0;
        } else {
            if (n <= kSortMax) key[s] = (ok && q1 > q0) ? (k1 - k0) : -1;
            tiles[s] = !ok ? 0 : bwd == 2 ? (heads / 2) * ((q1 - q0 + 127) / 128) : heads * ((q1 - q0 + 255) / 256);
        }
    }
    __syncthreads();
    for (int s = tid; s < n; s += kSchedThreads) {
        int rank = s;
        if (n <= kSortMax) {
            const int ks = key[s];
            rank = 0;
            for (int t = 0; t < n; ++t) {
                const int kt = key[t];
                rank += (kt > ks || (kt == ks && t < s)) ? 1 : 0;
            }
        }
        order[rank] = s;
    }
    __syncthreads();
    // exclusive scan of tiles in schedule order: per-thread chunks, then chunk offsets
    const int chunk = (n + kSchedThreads - 1) / kSchedThreads;
    const int c0 = min(n, tid * chunk), c1 = min(n, c0 + chunk);
    int sum = 0;
    for (int r = c0; r < c1; ++r) sum += tiles[order[r]];
    part[tid] = sum;
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int i = 0; i < kSchedThreads; ++i) {
            const int x = part[i];
            part[i] = acc;
            acc += x;
        }
        sched[0] = acc;
        prefix[n] = acc;
    }
    __syncthreads();
    int acc = part[tid];
    for (int r = c0; r < c1; ++r) {
        prefix[r] = acc;
        acc += tiles[order[r]];
    }
    if (bwd != 1) return;
    // padded row offsets in the original sequence order (valid sequences only)
    __syncthreads();
    int padded = 0;
    for (int s = c0; s < c1; ++s) padded += tiles[s] > 0 ? (cu_q[s + 1] - cu_q[s] + 127) / 128 * 128 : 0;
    part[tid] = padded;
    __syncthreads();
    if (tid == 0) {
        int a = 0;
        for (int i = 0; i < kSchedThreads; ++i) {
            const int x = part[i];
            part[i] = a;
            a += x;
        }
        sched[3 * n + 2 + n] = a;
    }
    __syncthreads();
    int* pad = sched + 3 * n + 2;
    int a = part[tid];
    for (int s = c0; s < c1; ++s) {
        pad[s] = a;
        a += tiles[s] > 0 ? (cu_q[s + 1] - cu_q[s] + 127) / 128 * 128 : 0;
    }
}

cudaError_t launch_varlen_schedule(const int* cu_q, const int* cu_k, int num_seqs, int total_q, int total_k,
                                   int max_q, int max_k, int heads, int bwd, int* sched, int* err,
                                   cudaStream_t stream)
{
    fa_varlen_schedule_kernel<<<1, kSchedThreads, 0, stream>>>(cu_q, cu_k, num_seqs, total_q, total_k, max_q,
                                                              max_k, heads, bwd, sched, err);
    return cudaGetLastError();
}

}  // namespace fa

using namespace fa;

namespace {
fa_status_t fwd_dense(const void* q, const void* k, const void* v, float* o, float* lse, int B, int Hq, int Hkv,
                      int Lq, int Lk, int D, int Dv, int causal, const fa_variant_t* variant, float softmax_scale,
                      cudaStream_t stream)
{
    g_last_launches = 0;
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0 || D <= 0 || Dv <= 0) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || !scale_ok(softmax_scale)) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_INVALID_ARG;
    if (!hdim_supported(D, Dv)) return FA_ERR_UNSUPPORTED;
    // causal GQA with an even group: work tiles of two query heads over 128 rows
    const bool pair = causal != 0 && !variant && (Hq / Hkv) % 2 == 0;
    const long long tiles = pair ? (long long)B * (Hq / 2) * ((Lq + kBlockM - 1) / kBlockM)
                                 : (long long)B * Hq * ((Lq + kRowsPerCta - 1) / kRowsPerCta);
    if (tiles >= (1ll << 31) || (long long)B * Hq >= (1ll << 31) || (long long)B * Hkv >= (1ll << 31))
        return FA_ERR_INVALID_ARG;
    FwdParams p{};
    int var = kVarNone;
    if (variant) {
        var = prepare_variant(variant, D, softmax_scale, &p);
        if (var < 0) return (fa_status_t)(-var);
        p.desc_tiles = window_tiles_desc(p, Lq, Lk);
    }
    DeviceState* ds = nullptr;
    fa_status_t st = device_state(&ds);
    if (st != FA_OK) return st;

    CUtensorMap mq, mk, mv;
    const uint64_t row = (uint64_t)D * 2, vrow = (uint64_t)Dv * 2;
    if (!encode_map(&mq, q, D, Lq, (uint64_t)B * Hq, row, row * Lq, 128, 1) ||
        !encode_map(&mk, k, D, Lk, (uint64_t)B * Hkv, row, row * Lk, 128, 1) ||
        !encode_map(&mv, v, Dv, Lk, (uint64_t)B * Hkv, vrow, vrow * Lk, 128, 1))
        return FA_ERR_CUDA;

    p.o = o;
    p.lse = lse;
    set_batch_heads(&p, B, Hq, Hkv, !var_alibi(var));
    p.Lq = Lq;
    p.Lk = Lk;
    p.group = Hq / Hkv;
    p.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);
    p.heads_per_section = heads_per_section(p.Hkv, Lk, D + Dv, !causal && var == kVarNone);
    p.num_tiles = (int)tiles;
    p.pair_heads = pair ? 1 : 0;
    p.err = ds->err;
    p.diag = ds->diag;
    p.fault = g_fault_next;
    g_fault_next = 0;
    const int grid = (int)(tiles < ds->num_sms ? tiles : ds->num_sms);
    const cudaError_t e = variant ? dispatch_variant<false>(D, var, mq, mk, mv, p, grid, stream)
                                  : dispatch<false>(D, causal != 0, mq, mk, mv, p, grid, stream);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    g_last_launches = 1;
    return FA_OK;
}
}  // namespace

extern "C" fa_status_t fa_fwd(const void* q, const void* k, const void* v, float* o, float* lse, int B, int Hq,
                              int Hkv, int Lq, int Lk, int D, int causal, float softmax_scale,
                              cudaStream_t stream)
{
    return fwd_dense(q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, D, D, causal, nullptr, softmax_scale, stream);
}

extern "C" fa_status_t fa_fwd_hdim(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                                   int Hq, int Hkv, int Lq, int Lk, int D, int Dv, int causal,
                                   float softmax_scale, cudaStream_t stream)
{
    return fwd_dense(q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, D, Dv, causal, nullptr, softmax_scale, stream);
}

extern "C" fa_status_t fa_fwd_variant(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                                      int Hq, int Hkv, int Lq, int Lk, int D, const fa_variant_t* variant,
                                      float softmax_scale, cudaStream_t stream)
{
    if (!variant) return FA_ERR_INVALID_ARG;
    return fwd_dense(q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, D, D, 0, variant, softmax_scale, stream);
}

// ------------------------------------------------------------- allocation-free varlen

// Scratch of fa_fwd_varlen_noalloc: the sequence schedule lives in this
// fixed device array instead of memory obtained per call.  Every GPU that
// loads the library holds it until the process exits.
constexpr int kNoAllocMaxSeqs = FA_NOALLOC_MAX_SEQS;
__device__ __align__(256) int g_noalloc_sched[2 + 3 * kNoAllocMaxSeqs];

namespace {
int* g_noalloc_ptr[kMaxDevices];  // device address of g_noalloc_sched, per device

// Resolves the array's device address on the current device (once per
// device).  In host code the symbol names a host-side stand-in, so only the
// address obtained here may be handed to a kernel.
fa_status_t noalloc_scratch(int** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_sched) != cudaSuccess || !ptr) return FA_ERR_CUDA;
        g_noalloc_ptr[dev] = static_cast<int*>(ptr);
    }
    *out = g_noalloc_ptr[dev];
    return FA_OK;
}
}  // namespace

namespace {
// Packed forward.  The library allocates nothing: normally each launch's CTAs
// build the schedule of up to varlen_sched_max_seqs(D, Dv) sequences in
// shared memory, and a larger batch is split into consecutive launches of
// that many sequences.  With `fixed_scratch` a schedule kernel writes one
// schedule for the whole batch into the library's fixed device array
// (g_noalloc_sched, at most FA_NOALLOC_MAX_SEQS sequences) and a single
// attention launch reads it.
fa_status_t fwd_varlen(const void* q, const void* k, const void* v, float* o, float* lse, const int* cu_seqlens_q,
                       const int* cu_seqlens_k, int num_seqs, int total_q, int total_k, int max_seqlen_q,
                       int max_seqlen_k, int Hq, int Hkv, int D, int Dv, int causal, const fa_variant_t* variant,
                       float softmax_scale, cudaStream_t stream, bool fixed_scratch = false)
{
    g_last_launches = 0;
    if (!q || !k || !v || !o || !lse || !cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID_ARG;
    if (num_seqs <= 0 || total_q <= 0 || total_k <= 0 || max_seqlen_q <= 0 || max_seqlen_k <= 0 || Hq <= 0 ||
        Hkv <= 0 || D <= 0 || Dv <= 0)
        return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || !scale_ok(softmax_scale)) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
        (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
        return FA_ERR_INVALID_ARG;
    if (!hdim_supported(D, Dv)) return FA_ERR_UNSUPPORTED;
    // work tiles: sum_s ceil(Lq_s / 256) <= total_q / 256 + num_seqs per query head
    if ((long long)Hq * ((long long)total_q / kRowsPerCta + num_seqs) >= (1ll << 31) ||
        (long long)total_q * Hq >= (1ll << 31) * 64ll)
        return FA_ERR_INVALID_ARG;
    FwdParams p{};
    int var = kVarNone;
    if (variant) {
        var = prepare_variant(variant, D, softmax_scale, &p);
        if (var < 0) return (fa_status_t)(-var);
        p.desc_tiles = window_tiles_desc(p, max_seqlen_q, max_seqlen_k);  // the longest sequence's profile
    }
    if (fixed_scratch && num_seqs > kNoAllocMaxSeqs) return FA_ERR_INVALID_ARG;  // the fixed array holds no more
    DeviceState* ds = nullptr;
    fa_status_t st = device_state(&ds);
    if (st != FA_OK) return st;
    int* sched_scratch = nullptr;
    if (fixed_scratch && (st = noalloc_scratch(&sched_scratch)) != FA_OK) return st;

    CUtensorMap mq, mk, mv;
    const uint64_t row = (uint64_t)D * 2, vrow = (uint64_t)Dv * 2;
    if (!encode_map(&mq, q, D, Hq, total_q, row, row * Hq, 1, 128) ||
        !encode_map(&mk, k, D, Hkv, total_k, row, row * Hkv, 1, 128) ||
        !encode_map(&mv, v, Dv, Hkv, total_k, vrow, vrow * Hkv, 1, 128))
        return FA_ERR_CUDA;

    p.o = o;
    p.lse = lse;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.group = Hq / Hkv;
    p.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);
    p.heads_per_section = heads_per_section(Hkv, max_seqlen_k, D + Dv, false);
    // causal GQA with an even group: work tiles of two query heads over 128 rows
    p.pair_heads = (causal != 0 && !variant && (Hq / Hkv) % 2 == 0) ? 1 : 0;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.num_seqs = num_seqs;
    p.total_q = total_q;
    p.total_k = total_k;
    p.max_q = max_seqlen_q;
    p.max_k = max_seqlen_k;
    p.err = ds->err;
    p.diag = ds->diag;
    const long long mb_per_seq = (max_seqlen_q + kRowsPerCta - 1) / kRowsPerCta;
    auto launch = [&](int count) -> cudaError_t {
        // grid: no more CTAs than work tiles can exist, at most one per SM
        long long ub = (long long)Hq * ((long long)total_q / kRowsPerCta + count);
        const long long ub2 = (long long)Hq * count * mb_per_seq;
        if (ub2 < ub) ub = ub2;
        const int grid = (int)(ub < ds->num_sms ? (ub > 0 ? ub : 1) : ds->num_sms);
        return variant ? dispatch_variant<true>(D, var, mq, mk, mv, p, grid, stream)
                       : dispatch<true>(D, causal != 0, mq, mk, mv, p, grid, stream);
    };
    if (sched_scratch) {
        if (launch_varlen_schedule(cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k, max_seqlen_q,
                                   max_seqlen_k, Hq, p.pair_heads ? 2 : 0, sched_scratch, ds->err, stream) !=
            cudaSuccess)
            return FA_ERR_CUDA;
        g_last_launches = 1;
        p.sched = sched_scratch;
        p.seq_begin = 0;
        p.seq_count = num_seqs;
        if (launch(num_seqs) != cudaSuccess) return FA_ERR_CUDA;
        g_last_launches = 2;
        return FA_OK;
    }
    static_assert(varlen_sched_max_seqs(64, 64) == FA_VARLEN_SEQS_PER_LAUNCH &&
                      varlen_sched_max_seqs(128, 128) == FA_VARLEN_SEQS_PER_LAUNCH,
                  "launch size of packed batches differs from the header's");
    const int per_launch = varlen_sched_max_seqs(D, Dv);
    for (int b = 0; b < num_seqs; b += per_launch) {
        p.sched = nullptr;
        p.seq_begin = b;
        p.seq_count = num_seqs - b < per_launch ? num_seqs - b : per_launch;
        if (launch(p.seq_count) != cudaSuccess) return FA_ERR_CUDA;
        ++g_last_launches;
    }
    return FA_OK;
}
}  // namespace

extern "C" fa_status_t fa_fwd_varlen(const void* q, const void* k, const void* v, float* o, float* lse,
                                     const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs,
                                     int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int Hq,
                                     int Hkv, int D, int causal, float softmax_scale, cudaStream_t stream)
{
    return fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k, max_seqlen_q,
                      max_seqlen_k, Hq, Hkv, D, D, causal, nullptr, softmax_scale, stream);
}

extern "C" fa_status_t fa_fwd_varlen_hdim(const void* q, const void* k, const void* v, float* o, float* lse,
                                          const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs,
                                          int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int Hq,
                                          int Hkv, int D, int Dv, int causal, float softmax_scale,
                                          cudaStream_t stream)
{
    return fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k, max_seqlen_q,
                      max_seqlen_k, Hq, Hkv, D, Dv, causal, nullptr, softmax_scale, stream);
}

extern "C" fa_status_t fa_fwd_varlen_variant(const void* q, const void* k, const void* v, float* o, float* lse,
                                             const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs,
                                             int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                                             int Hq, int Hkv, int D, const fa_variant_t* variant,
                                             float softmax_scale, cudaStream_t stream)
{
    if (!variant) return FA_ERR_INVALID_ARG;
    return fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k, max_seqlen_q,
                      max_seqlen_k, Hq, Hkv, D, D, 0, variant, softmax_scale, stream);
}

extern "C" fa_status_t fa_fwd_varlen_noalloc(const void* q, const void* k, const void* v, float* o, float* lse,
                                             const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs,
                                             int total_q, int total_k, int max_seqlen_q, int max_seqlen_k,
                                             int Hq, int Hkv, int D, int causal, float softmax_scale,
                                             cudaStream_t stream)
{
    // The schedule kernel writes every scratch entry the attention kernel
    // reads, so nothing left by an earlier call needs clearing.
    return fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k, max_seqlen_q,
                      max_seqlen_k, Hq, Hkv, D, D, causal, nullptr, softmax_scale, stream, true);
}

// ------------------------------------------------------------- split-KV decode

namespace {

constexpr int kMaxSplits = 1024;

struct SplitPlan {
    int R = 0, rpt = 0, num_tiles = 0, splits = 1, tiles_per_split = 0;
    bool tensor = false;  // tensor-core partials (128-key tiles) instead of the FP32-pipe kernel
    size_t ws_bytes = 0;
};

fa_status_t splitkv_validate(int B, int Hq, int Hkv, int Lq, int Lk, int D)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0 || D <= 0) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    if ((long long)(Hq / Hkv) * Lq > kDecMaxRows) return FA_ERR_UNSUPPORTED;
    if ((long long)B * Hq * Lq >= (1ll << 31) || (long long)B * Hkv >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    return FA_OK;
}

// Partitions of the key range.  The pages leave the count to the workload:
// more partitions fill more SMs but add partial results and a merge.  The
// automatic choice minimises a small cost model in units of one tile per CTA
// slot: waves of work items over the GPU's resident slots times the tiles of
// one partition (+2 for pipeline fill), plus the merge (a launch and the
// partial-result bytes spread over the whole GPU).
void splitkv_plan(int B, int Hq, int Hkv, int Lq, int Lk, int D, int num_splits, int num_sms, SplitPlan* pl)
{
    pl->R = (Hq / Hkv) * Lq;
    pl->tensor = (D == 64 || D == 128) && pl->R >= 2;
    pl->rpt = decode_rows_per_thread(D, pl->R);
    const int keys = pl->tensor ? decode_tc_keys(D) : kDecKeys;
    pl->num_tiles = (Lk + keys - 1) / keys;
    const int nkt = pl->num_tiles;
    const long long bh = (long long)B * Hkv;
    int splits = 1;
    if (num_splits > 0) {
        splits = num_splits < nkt ? num_splits : nkt;
    } else {
        const long long slots = (long long)num_sms * (pl->tensor ? 1 : decode_ctas_per_sm(D, pl->rpt));
        const double tile_bytes = 2.0 * keys * D * 2;
        double best = 1e300;
        for (int s = 1; s <= nkt && s <= kMaxSplits; ++s) {
            const int tps = (nkt + s - 1) / s;
            if ((nkt + tps - 1) / tps != s) continue;  // same partition as a smaller count
            if (bh * s >= (1ll << 31)) break;
            const long long waves = (bh * s + slots - 1) / slots;
            double cost = (double)waves * (tps + 2.0);
            if (s > 1) cost += 2.0 + (double)bh * s * pl->R * (D + 1) * 8.0 / ((double)slots * tile_bytes);
            if (cost < best * (1.0 - 1e-9)) {
                best = cost;
                splits = s;
            }
        }
    }
    pl->tiles_per_split = (nkt + splits - 1) / splits;
    pl->splits = (nkt + pl->tiles_per_split - 1) / pl->tiles_per_split;  // no empty partition
    pl->ws_bytes = 0;
    if (pl->splits > 1) {
        const size_t rows = (size_t)bh * pl->splits * pl->R;
        pl->ws_bytes = ((rows * D + rows) * sizeof(float) + 255) & ~(size_t)255;
    }
}

}  // namespace

extern "C" fa_status_t fa_fwd_splitkv_workspace(int B, int Hq, int Hkv, int Lq, int Lk, int D, int num_splits,
                                                size_t* workspace_bytes, int* splits_used)
{
    if (!workspace_bytes) return FA_ERR_INVALID_ARG;
    fa_status_t st = splitkv_validate(B, Hq, Hkv, Lq, Lk, D);
    if (st != FA_OK) return st;
    DeviceState* ds = nullptr;
    st = device_state(&ds);
    if (st != FA_OK) return st;
    SplitPlan pl;
    splitkv_plan(B, Hq, Hkv, Lq, Lk, D, num_splits, ds->num_sms, &pl);
    if ((long long)B * Hkv * pl.splits >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    *workspace_bytes = pl.ws_bytes;
    if (splits_used) *splits_used = pl.splits;
    return FA_OK;
}

extern "C" fa_status_t fa_fwd_splitkv(const void* q, const void* k, const void* v, float* o, float* lse, int B,
                                      int Hq, int Hkv, int Lq, int Lk, int D, int causal, float softmax_scale,
                                      int num_splits, void* workspace, size_t workspace_bytes,
                                      cudaStream_t stream)
{
    g_last_launches = 0;
    if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
    fa_status_t st = splitkv_validate(B, Hq, Hkv, Lq, Lk, D);
    if (st != FA_OK) return st;
    if (!scale_ok(softmax_scale)) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return FA_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    st = device_state(&ds);
    if (st != FA_OK) return st;
    SplitPlan pl;
    splitkv_plan(B, Hq, Hkv, Lq, Lk, D, num_splits, ds->num_sms, &pl);
    const long long grid = (long long)B * Hkv * pl.splits;
    if (pl.rpt == 0 || grid >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    if (pl.ws_bytes > 0 && (!workspace || !aligned16(workspace) || workspace_bytes < pl.ws_bytes))
        return FA_ERR_INVALID_ARG;

    CUtensorMap mq, mk, mv;
    const uint64_t row = (uint64_t)D * 2;
    const uint32_t box_keys = pl.tensor ? kDecTcKeys : kDecKeys;
    if (!encode_map(&mk, k, D, Lk, (uint64_t)B * Hkv, row, row * Lk, box_keys, 1) ||
        !encode_map(&mv, v, D, Lk, (uint64_t)B * Hkv, row, row * Lk, box_keys, 1))
        return FA_ERR_CUDA;
    const uint64_t q_rows = (uint64_t)B * Hq * Lq;
    if (pl.tensor && !encode_map(&mq, q, D, q_rows, 1, row, row * q_rows, kDecMaxRows, 1)) return FA_ERR_CUDA;

    DecodeParams p{};
    p.q = static_cast<const uint16_t*>(q);
    p.o = o;
    p.lse = lse;
    if (pl.splits > 1) {
        const size_t rows = (size_t)grid * pl.R;
        p.o_part = static_cast<float*>(workspace);
        p.l_part = p.o_part + rows * D;
    }
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Lq = Lq;
    p.Lk = Lk;
    p.group = Hq / Hkv;
    p.R = pl.R;
    p.num_splits = pl.splits;
    p.tiles_per_split = pl.tiles_per_split;
    p.num_tiles = pl.num_tiles;
    p.causal = causal != 0;
    p.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);
    p.err = ds->err;
    p.diag = ds->diag;
    p.fault = g_fault_next;
    g_fault_next = 0;
    if (pl.tensor) {
        const int g = (int)(grid < ds->num_sms ? grid : ds->num_sms);
        if (launch_decode_tc(D, mq, mk, mv, p, g, stream) != cudaSuccess) return FA_ERR_CUDA;
    } else if (launch_decode_partial(D, pl.rpt, mk, mv, p, (int)grid, stream) != cudaSuccess) {
        return FA_ERR_CUDA;
    }
    if (pl.splits > 1 && launch_decode_merge(D, p, stream) != cudaSuccess) return FA_ERR_CUDA;
    g_last_launches = pl.splits > 1 ? 2 : 1;
    return FA_OK;
}

// ------------------------------------------------------------- backward

namespace {
long long bwd_rows_padded(int Lq) { return ((long long)Lq + kBwdTile - 1) / kBwdTile * kBwdTile; }

// (batch, KV head) slabs per scheduling section of the backward: the dQ
// (fp32), Q and dO (bf16) of a section's query heads, 8 * D bytes per query
// row, should fit in half of the L2.  Sections break the longest-first
// order of the item list, so they are used only when every CTA gets many
// items (measured: with about 3 items per CTA, a causal GQA problem lost a
// quarter of its speed to imbalance).
int bwd_heads_per_section(int slabs, int group, long long Lq, int D, long long items, int num_sms)
{
    constexpr long long kBudget = 64ll << 20;
    if (items < 8ll * num_sms) return slabs;
    const long long per = (long long)group * Lq * 8 * D;
    long long hs = per > 0 ? kBudget / per : slabs;
    if (hs < 1) hs = 1;
    if (hs > slabs) hs = slabs;
    return (int)hs;
}
}  // namespace

extern "C" fa_status_t fa_bwd_workspace(int B, int Hq, int Lq, size_t* workspace_bytes)
{
    if (!workspace_bytes || B <= 0 || Hq <= 0 || Lq <= 0) return FA_ERR_INVALID_ARG;
    const long long rows = (long long)B * Hq * bwd_rows_padded(Lq);
    if (rows >= (1ll << 40)) return FA_ERR_INVALID_ARG;
    *workspace_bytes = (size_t)((2 * rows * (long long)sizeof(float) + 255) & ~255ll);
    return FA_OK;
}

namespace {
// Validates a backward variant (windows, soft-capping, ALiBi; soft-capping
// and ALiBi together are unsupported, as in the forward) and fills the
// parameters; returns the variant kind or a negative fa_status_t.
int prepare_bwd_variant(const fa_variant_t* var, int D, float scale, BwdParams* p)
{
    if (!var) return -(int)FA_ERR_INVALID_ARG;
    if (!std::isfinite(var->softcap) || var->softcap < 0.f) return -(int)FA_ERR_INVALID_ARG;
    if (var->alibi_slopes && (reinterpret_cast<uintptr_t>(var->alibi_slopes) & 3u)) return -(int)FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return -(int)FA_ERR_UNSUPPORTED;
    p->win_left = var->window_left < 0 ? -1 : var->window_left;
    p->win_right = var->window_right < 0 ? -1 : var->window_right;
    p->alibi = var->alibi_slopes;
    if (var->softcap > 0.f) {
        p->cap_in2 = (float)(2.0 * 1.4426950408889634 * (double)scale / (double)var->softcap);
        p->cap_out = (float)((double)var->softcap * 1.4426950408889634);
        return var->alibi_slopes ? kVarCapAlibi : kVarSoftcap;
    }
    return var->alibi_slopes ? kVarAlibi : kVarWindow;
}

fa_status_t bwd_dense(const void* q, const void* k, const void* v, const float* o, const float* lse,
                      const void* dout, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int Lq, int Lk,
                      int D, int causal, const fa_variant_t* variant, float softmax_scale, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream)
{
    g_last_launches = 0;
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0 || D <= 0) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || !scale_ok(softmax_scale)) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
        return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    const long long lq_pad = bwd_rows_padded(Lq);
    const long long rows = (long long)B * Hq * lq_pad;
    if (rows >= (1ll << 31) || (long long)B * Hq >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    const long long kv_tiles = ((long long)Lk + kBwdTile - 1) / kBwdTile;
    const long long items = (long long)B * Hkv * kv_tiles;
    if (items >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    size_t need = 0;
    fa_bwd_workspace(B, Hq, Lq, &need);
    if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
    BwdParams p{};
    int var = kVarNone;
    if (variant) {
        var = prepare_bwd_variant(variant, D, softmax_scale, &p);
        if (var < 0) return (fa_status_t)(-var);
    }
    DeviceState* ds = nullptr;
    fa_status_t st = device_state(&ds);
    if (st != FA_OK) return st;

    CUtensorMap mq, mk, mv, mdo;
    const uint64_t row = (uint64_t)D * 2;
    if (!encode_map(&mq, q, D, Lq, (uint64_t)B * Hq, row, row * Lq, kBwdTile, 1) ||
        !encode_map(&mdo, dout, D, Lq, (uint64_t)B * Hq, row, row * Lq, kBwdTile, 1) ||
        !encode_map(&mk, k, D, Lk, (uint64_t)B * Hkv, row, row * Lk, kBwdTile, 1) ||
        !encode_map(&mv, v, D, Lk, (uint64_t)B * Hkv, row, row * Lk, kBwdTile, 1))
        return FA_ERR_CUDA;
    CUtensorMap mdq;  // dQ reduce-adds: [32 rows][32 columns] fp32 boxes
    if (!encode_map_f32(&mdq, dq, D, Lq, (uint64_t)B * Hq, (uint64_t)D * 4, (uint64_t)D * 4 * Lq, 32, 32, 1))
        return FA_ERR_CUDA;

    p.o = o;
    p.lse = lse;
    p.dout = static_cast<const uint16_t*>(dout);
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.delta = static_cast<float*>(workspace);
    p.lse2 = p.delta + rows;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Lq = Lq;
    p.Lk = Lk;
    p.Lq_pad = (int)lq_pad;
    p.group = Hq / Hkv;
    p.num_kv_tiles = (int)kv_tiles;
    p.num_q_tiles = (int)(lq_pad / kBwdTile);
    p.num_items = (int)items;
    p.heads_per_section = bwd_heads_per_section(B * Hkv, Hq / Hkv, Lq, D, items, ds->num_sms);
    p.scale = softmax_scale;
    p.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);
    p.causal = causal != 0;
    p.err = ds->err;
    p.diag = ds->diag;
    p.fault = g_fault_next;
    g_fault_next = 0;
    if (launch_bwd_pre(D, false, p, stream) != cudaSuccess) return FA_ERR_CUDA;
    const int grid = (int)(items < ds->num_sms ? items : ds->num_sms);
    const cudaError_t e = variant ? launch_bwd_variant(D, var, false, mq, mk, mv, mdo, mdq, p, grid, stream)
                                  : launch_bwd(D, causal != 0, false, mq, mk, mv, mdo, mdq, p, grid, stream);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    g_last_launches = 2;
    return FA_OK;
}
}  // namespace

extern "C" fa_status_t fa_bwd(const void* q, const void* k, const void* v, const float* o, const float* lse,
                              const void* dout, float* dq, float* dk, float* dv, int B, int Hq, int Hkv, int Lq,
                              int Lk, int D, int causal, float softmax_scale, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream)
{
    return bwd_dense(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Lq, Lk, D, causal, nullptr, softmax_scale,
                     workspace, workspace_bytes, stream);
}

extern "C" fa_status_t fa_bwd_variant(const void* q, const void* k, const void* v, const float* o,
                                      const float* lse, const void* dout, float* dq, float* dk, float* dv, int B,
                                      int Hq, int Hkv, int Lq, int Lk, int D, const fa_variant_t* variant,
                                      float softmax_scale, void* workspace, size_t workspace_bytes,
                                      cudaStream_t stream)
{
    if (!variant) return FA_ERR_INVALID_ARG;
    return bwd_dense(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Lq, Lk, D, 0, variant, softmax_scale,
                     workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------- packed backward

namespace {
// Workspace of fa_bwd_varlen: delta and lse2 as [Hq][rows], every sequence's
// rows padded to a multiple of 128 (rows = an upper bound of the padded total),
// then the schedule (4 * num_seqs + 3 ints).
struct BwdVarlenLayout {
    long long rows = 0;
    size_t sched_off = 0, bytes = 0;
};

bool bwd_varlen_layout(int num_seqs, int total_q, int Hq, BwdVarlenLayout* l)
{
    if (num_seqs <= 0 || total_q <= 0 || Hq <= 0) return false;
    l->rows = ((long long)total_q + 127) / 128 * 128 + 128ll * num_seqs;
    const long long floats = 2ll * Hq * l->rows;
    if (floats >= (1ll << 40)) return false;
    l->sched_off = (size_t)((floats * 4 + 255) & ~255ll);
    l->bytes = (l->sched_off + sizeof(int) * (4 * (size_t)num_seqs + 3) + 255) & ~(size_t)255;
    return true;
}
}  // namespace

extern "C" fa_status_t fa_bwd_varlen_workspace(int num_seqs, int total_q, int Hq, size_t* workspace_bytes)
{
    BwdVarlenLayout l;
    if (!workspace_bytes || !bwd_varlen_layout(num_seqs, total_q, Hq, &l)) return FA_ERR_INVALID_ARG;
    *workspace_bytes = l.bytes;
    return FA_OK;
}

namespace {
fa_status_t bwd_varlen(const void* q, const void* k, const void* v, const float* o, const float* lse,
                       const void* dout, float* dq, float* dk, float* dv, const int* cu_seqlens_q,
                       const int* cu_seqlens_k, int num_seqs, int total_q, int total_k, int max_seqlen_q,
                       int max_seqlen_k, int Hq, int Hkv, int D, int causal, const fa_variant_t* variant,
                       float softmax_scale, void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    g_last_launches = 0;
    if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace || !cu_seqlens_q ||
        !cu_seqlens_k)
        return FA_ERR_INVALID_ARG;
    if (num_seqs <= 0 || total_q <= 0 || total_k <= 0 || max_seqlen_q <= 0 || max_seqlen_k <= 0 || Hq <= 0 ||
        Hkv <= 0 || D <= 0)
        return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0 || !scale_ok(softmax_scale)) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
        return FA_ERR_INVALID_ARG;
    if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    BwdVarlenLayout lay;
    if (!bwd_varlen_layout(num_seqs, total_q, Hq, &lay) || workspace_bytes < lay.bytes) return FA_ERR_INVALID_ARG;
    // upper bound of the work items: sum_s ceil(Lk_s / 128) <= total_k / 128 + num_seqs
    const long long ub = (long long)Hkv * ((long long)total_k / kBwdTile + num_seqs);
    if (ub >= (1ll << 31) || lay.rows >= (1ll << 31) || (long long)total_q * Hq >= (1ll << 31) * 8ll ||
        (long long)total_k * Hkv >= (1ll << 31) * 8ll)
        return FA_ERR_INVALID_ARG;
    BwdParams p{};
    int var = kVarNone;
    if (variant) {
        var = prepare_bwd_variant(variant, D, softmax_scale, &p);
        if (var < 0) return (fa_status_t)(-var);
    }
    DeviceState* ds = nullptr;
    fa_status_t st = device_state(&ds);
    if (st != FA_OK) return st;

    CUtensorMap mq, mk, mv, mdo;
    const uint64_t row = (uint64_t)D * 2;
    if (!encode_map(&mq, q, D, Hq, total_q, row, row * Hq, 1, kBwdTile) ||
        !encode_map(&mdo, dout, D, Hq, total_q, row, row * Hq, 1, kBwdTile) ||
        !encode_map(&mk, k, D, Hkv, total_k, row, row * Hkv, 1, kBwdTile) ||
        !encode_map(&mv, v, D, Hkv, total_k, row, row * Hkv, 1, kBwdTile))
        return FA_ERR_CUDA;
    CUtensorMap mdq;  // dQ reduce-adds: [32 tokens][1 head][32 columns] fp32 boxes
    if (!encode_map_f32(&mdq, dq, D, Hq, total_q, (uint64_t)D * 4, (uint64_t)D * 4 * Hq, 32, 1, 32))
        return FA_ERR_CUDA;

    int* sched = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + lay.sched_off);
    if (launch_varlen_schedule(cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k, max_seqlen_q,
                               max_seqlen_k, Hkv, 1, sched, ds->err, stream) != cudaSuccess)
        return FA_ERR_CUDA;
    p.o = o;
    p.lse = lse;
    p.dout = static_cast<const uint16_t*>(dout);
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.delta = static_cast<float*>(workspace);
    p.lse2 = p.delta + (long long)Hq * lay.rows;
    p.B = 1;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Lq_pad = (int)lay.rows;
    p.group = Hq / Hkv;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.sched = sched;
    p.num_seqs = num_seqs;
    p.total_q = total_q;
    p.total_k = total_k;
    p.heads_per_section = bwd_heads_per_section(Hkv, Hq / Hkv, max_seqlen_q, D, ub, ds->num_sms);
    p.scale = softmax_scale;
    p.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);
    p.causal = causal != 0;
    p.err = ds->err;
    p.diag = ds->diag;
    p.fault = g_fault_next;
    g_fault_next = 0;
    if (launch_bwd_pre(D, true, p, stream) != cudaSuccess) return FA_ERR_CUDA;
    const int grid = (int)(ub < ds->num_sms ? (ub > 0 ? ub : 1) : ds->num_sms);
    const cudaError_t e = variant ? launch_bwd_variant(D, var, true, mq, mk, mv, mdo, mdq, p, grid, stream)
                                  : launch_bwd(D, causal != 0, true, mq, mk, mv, mdo, mdq, p, grid, stream);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    g_last_launches = 3;
    return FA_OK;
}
}  // namespace

extern "C" fa_status_t fa_bwd_varlen(const void* q, const void* k, const void* v, const float* o, const float* lse,
                                     const void* dout, float* dq, float* dk, float* dv, const int* cu_seqlens_q,
                                     const int* cu_seqlens_k, int num_seqs, int total_q, int total_k,
                                     int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D, int causal,
                                     float softmax_scale, void* workspace, size_t workspace_bytes,
                                     cudaStream_t stream)
{
    return bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k,
                      max_seqlen_q, max_seqlen_k, Hq, Hkv, D, causal, nullptr, softmax_scale, workspace,
                      workspace_bytes, stream);
}

extern "C" fa_status_t fa_bwd_varlen_variant(const void* q, const void* k, const void* v, const float* o,
                                             const float* lse, const void* dout, float* dq, float* dk, float* dv,
                                             const int* cu_seqlens_q, const int* cu_seqlens_k, int num_seqs,
                                             int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int Hq,
                                             int Hkv, int D, const fa_variant_t* variant, float softmax_scale,
                                             void* workspace, size_t workspace_bytes, cudaStream_t stream)
{
    if (!variant) return FA_ERR_INVALID_ARG;
    return bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k,
                      max_seqlen_q, max_seqlen_k, Hq, Hkv, D, 0, variant, softmax_scale, workspace, workspace_bytes,
                      stream);
}

// ------------------------------------------------------------- FP8 forward

namespace {

// Sections of a prepared FP8 buffer, each 256-byte aligned.
struct Fp8Layout {
    size_t qc, kc, vt, sq, sk, sv, vmax, total;
    int nq, nk, lk_pad;
};

bool fp8_layout(int B, int Hq, int Hkv, int Lq, int Lk, Fp8Layout* l)
{
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    l->nq = (Lq + kFp8Tile - 1) / kFp8Tile;
    l->nk = (Lk + kFp8Tile - 1) / kFp8Tile;
    l->lk_pad = l->nk * kFp8Tile;
    size_t off = 0;
    l->qc = off; off = up(off + (size_t)B * Hq * Lq * 128);
    l->kc = off; off = up(off + (size_t)B * Hkv * Lk * 128);
    l->vt = off; off = up(off + (size_t)B * Hkv * 128 * l->lk_pad);
    l->sq = off; off = up(off + (size_t)B * Hq * l->nq * 4);
    l->sk = off; off = up(off + (size_t)B * Hkv * l->nk * 4);
    l->sv = off; off = up(off + (size_t)B * Hkv * 4);
    l->vmax = off; off = up(off + (size_t)B * Hkv * 4);
    l->total = off;
    return true;
}

fa_status_t fp8_validate(int B, int Hq, int Hkv, int Lq, int Lk, int D)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lk <= 0 || D <= 0) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
    if (D != 128) return FA_ERR_UNSUPPORTED;
    if ((long long)B * Hq * Lq >= (1ll << 31) || (long long)B * Hkv * (Lk + kFp8Tile) >= (1ll << 31))
        return FA_ERR_INVALID_ARG;
    return FA_OK;
}

// 3-D e4m3 (byte) tensor map, 128-byte swizzle, box = {128, box1, 1}.
bool encode_map_u8(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1,
                   uint64_t stride2, uint32_t box1)
{
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1, stride2};
    const cuuint32_t box[3] = {128, box1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" fa_status_t fa_fp8_workspace(int B, int Hq, int Hkv, int Lq, int Lk, int D, size_t* bytes)
{
    if (!bytes) return FA_ERR_INVALID_ARG;
    const fa_status_t st = fp8_validate(B, Hq, Hkv, Lq, Lk, D);
    if (st != FA_OK) return st;
    Fp8Layout l;
    fp8_layout(B, Hq, Hkv, Lq, Lk, &l);
    *bytes = l.total;
    return FA_OK;
}

extern "C" fa_status_t fa_fp8_prepare(const void* q, const void* k, const void* v, const float* signs, int B,
                                      int Hq, int Hkv, int Lq, int Lk, int D, void* prepared,
                                      size_t prepared_bytes, cudaStream_t stream)
{
    g_last_launches = 0;
    if (!q || !k || !v || !signs || !prepared) return FA_ERR_INVALID_ARG;
    fa_status_t st = fp8_validate(B, Hq, Hkv, Lq, Lk, D);
    if (st != FA_OK) return st;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(prepared) ||
        (reinterpret_cast<uintptr_t>(signs) & 3u))
        return FA_ERR_INVALID_ARG;
    Fp8Layout l;
    fp8_layout(B, Hq, Hkv, Lq, Lk, &l);
    if (prepared_bytes < l.total) return FA_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    st = device_state(&ds);
    if (st != FA_OK) return st;
    uint8_t* base = static_cast<uint8_t*>(prepared);
    Fp8PrepParams p{};
    p.q = static_cast<const uint16_t*>(q);
    p.k = static_cast<const uint16_t*>(k);
    p.v = static_cast<const uint16_t*>(v);
    p.signs = signs;
    p.qc = base + l.qc;
    p.kc = base + l.kc;
    p.vt = base + l.vt;
    p.sq = reinterpret_cast<float*>(base + l.sq);
    p.sk = reinterpret_cast<float*>(base + l.sk);
    p.sv = reinterpret_cast<float*>(base + l.sv);
    p.vmax = reinterpret_cast<unsigned*>(base + l.vmax);
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Lq = Lq;
    p.Lk = Lk;
    p.Lk_pad = l.lk_pad;
    p.nq = l.nq;
    p.nk = l.nk;
    if (cudaMemsetAsync(p.vmax, 0, (size_t)B * Hkv * 4, stream) != cudaSuccess) return FA_ERR_CUDA;
    if (launch_fp8_prepare(p, stream) != cudaSuccess) return FA_ERR_CUDA;
    g_last_launches = 3;
    return FA_OK;
}

extern "C" fa_status_t fa_fwd_fp8(const void* prepared, float* o, float* lse, int B, int Hq, int Hkv, int Lq,
                                  int Lk, int D, int causal, float softmax_scale, cudaStream_t stream)
{
    g_last_launches = 0;
    if (!prepared || !o || !lse) return FA_ERR_INVALID_ARG;
    fa_status_t st = fp8_validate(B, Hq, Hkv, Lq, Lk, D);
    if (st != FA_OK) return st;
    if (!scale_ok(softmax_scale)) return FA_ERR_INVALID_ARG;
    if (!aligned16(prepared) || !aligned16(o) || !aligned16(lse)) return FA_ERR_INVALID_ARG;
    const long long nmb = (Lq + kRowsPerCta - 1) / kRowsPerCta;
    const long long tiles = (long long)B * Hq * nmb;
    if (tiles >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    st = device_state(&ds);
    if (st != FA_OK) return st;
    Fp8Layout l;
    fp8_layout(B, Hq, Hkv, Lq, Lk, &l);
    const uint8_t* base = static_cast<const uint8_t*>(prepared);
    CUtensorMap mq, mk, mv;
    if (!encode_map_u8(&mq, base + l.qc, 128, Lq, (uint64_t)B * Hq, 128, 128ull * Lq, 128) ||
        !encode_map_u8(&mk, base + l.kc, 128, Lk, (uint64_t)B * Hkv, 128, 128ull * Lk, 128) ||
        !encode_map_u8(&mv, base + l.vt, l.lk_pad, 128, (uint64_t)B * Hkv, l.lk_pad, 128ull * l.lk_pad, 128))
        return FA_ERR_CUDA;
    FwdParams p{};
    p.o = o;
    p.lse = lse;
    set_batch_heads(&p, B, Hq, Hkv, true);  // the scales are indexed by (batch, head) slab
    p.Lq = Lq;
    p.Lk = Lk;
    p.group = Hq / Hkv;
    p.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);
    p.heads_per_section = heads_per_section(p.Hkv, Lk, D / 2, !causal);  // e4m3 K/V: half the bytes of bf16
    p.num_tiles = (int)tiles;
    p.fp8_sq = reinterpret_cast<const float*>(base + l.sq);
    p.fp8_sk = reinterpret_cast<const float*>(base + l.sk);
    p.fp8_sv = reinterpret_cast<const float*>(base + l.sv);
    p.fp8_nq = l.nq;
    p.fp8_nk = l.nk;
    p.err = ds->err;
    p.diag = ds->diag;
    p.fault = g_fault_next;
    g_fault_next = 0;
    const int grid = (int)(tiles < ds->num_sms ? tiles : ds->num_sms);
    const cudaError_t e = causal ? launch_fwd<128, true, false, kVarFp8>(mq, mk, mv, p, grid, stream)
                                 : launch_fwd<128, false, false, kVarFp8>(mq, mk, mv, p, grid, stream);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    g_last_launches = 1;
    return FA_OK;
}

extern "C" fa_status_t fa_check(cudaStream_t stream)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
    DeviceState* ds = nullptr;
    fa_status_t st = device_state(&ds);
    if (st != FA_OK) return st;
    int h = 0;
    if (cudaMemcpyFromSymbol(&h, g_err, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
    if (h == 0) return FA_OK;
    const int zero[4] = {0, 0, 0, 0};
    if (cudaMemcpyToSymbol(g_err, zero, sizeof(int)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_diag, zero, sizeof(zero)) != cudaSuccess)
        return FA_ERR_CUDA;
    if (h & 1) return FA_ERR_TIMEOUT;
    return (h & 4) ? FA_ERR_CUDA : FA_ERR_INVALID_ARG;
}

extern "C" const char* fa_status_string(fa_status_t s)
{
    switch (s) {
        case FA_OK: return "ok";
        case FA_ERR_INVALID_ARG: return "invalid argument";
        case FA_ERR_UNSUPPORTED: return "unsupported configuration";
        case FA_ERR_CUDA: return "CUDA error";
        case FA_ERR_TIMEOUT: return "kernel pipeline wait timed out";
    }
    return "unknown status";
}

extern "C" int fa_last_launch_count(void) { return g_last_launches; }

extern "C" void fa_test_inject_fault(int kind) { g_fault_next = kind; }
