// Attention backward: parameters and host launch entry points.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include <cstdint>

#include "fa_params.h"

namespace fa {

constexpr int kBwdTile = 128;  // keys per KV tile = query rows per Q tile

// Dense layouts are [B, H, L, D]; packed (varlen) ones [T, H, D] with LSE
// [Hq, Tq], as in the forward.
struct BwdParams {
    // preprocess inputs
    const float* o;         // forward output (fp32)
    const float* lse;       // forward LSE, natural log
    const uint16_t* dout;   // bf16, layout of Q
    // outputs (fp32)
    float* dq;              // layout of Q; zeroed by the preprocess kernel, then accumulated
    float* dk;              // layout of K
    float* dv;              // layout of V
    // workspace, [B * Hq][Lq_pad] each (varlen: [Hq][Lq_pad], every sequence's
    // rows padded to a multiple of 128, starting at its padded row offset)
    float* delta;           // rowsum(O * dO); 0 on padding rows
    float* lse2;            // LSE * log2(e); +inf on rows without keys and on padding rows
    int B, Hq, Hkv, Lq, Lk, Lq_pad, group;
    // packed batches: sequence offsets (int32, device) and the schedule built
    // by the varlen schedule kernel (item prefix, order, items by sequence,
    // padded row offsets)
    const int* cu_q;
    const int* cu_k;
    const int* sched;
    int num_seqs, total_q, total_k;
    int num_kv_tiles;       // ceil(Lk / 128)
    int num_q_tiles;        // ceil(Lq / 128)
    int num_items;          // B * Hkv * num_kv_tiles
    int heads_per_section;  // (batch, KV head) slabs whose items are interleaved (L2-sized dQ working set)
    // variants (kernels instantiated with VAR > 0): key window around each
    // query's aligned position (< 0 = unlimited) and ALiBi slopes per query
    // head (natural-log units)
    int win_left, win_right;
    const float* alibi;
    // soft-capping (VAR = kVarSoftcap): 2 log2(e) scale / cap and cap log2(e)
    float cap_in2, cap_out;
    float scale;            // softmax_scale (multiplies dS)
    float scale_log2;       // softmax_scale * log2(e)
    int causal;
    int* err;
    int* diag;
    int fault;              // test hook: 1 = skip the first K/V load of every CTA
};

cudaError_t launch_bwd_pre(int D, bool varlen, const BwdParams& p, cudaStream_t stream);
// dq: fp32 tensor map of dQ with 128-byte swizzle, box {32, 32, 1} (dense) or
// {32, 1, 32} (packed);
// used at D = 128.
cudaError_t launch_bwd(int D, bool causal, bool varlen, const CUtensorMap& q, const CUtensorMap& k,
                       const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& dq, const BwdParams& p,
                       int grid, cudaStream_t stream);
// Variants (var = kVarWindow, kVarSoftcap, kVarAlibi or kVarCapAlibi, no separate causal
// flag: a causal window is (-1, 0)), head dimension 64 or 128, each in a
// translation unit of its own.
cudaError_t launch_bwd_variant_d64(int var, bool varlen, const CUtensorMap& q, const CUtensorMap& k,
                                   const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& dq,
                                   const BwdParams& p, int grid, cudaStream_t stream);
cudaError_t launch_bwd_variant_d128(int var, bool varlen, const CUtensorMap& q, const CUtensorMap& k,
                                    const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& dq,
                                    const BwdParams& p, int grid, cudaStream_t stream);
inline cudaError_t launch_bwd_variant(int D, int var, bool varlen, const CUtensorMap& q, const CUtensorMap& k,
                                      const CUtensorMap& v, const CUtensorMap& dout, const CUtensorMap& dq,
                                      const BwdParams& p, int grid, cudaStream_t stream)
{
    if (D == 64) return launch_bwd_variant_d64(var, varlen, q, k, v, dout, dq, p, grid, stream);
    if (D == 128) return launch_bwd_variant_d128(var, varlen, q, k, v, dout, dq, p, grid, stream);
    return cudaErrorInvalidValue;
}

}  // namespace fa
