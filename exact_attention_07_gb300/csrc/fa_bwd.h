// Attention backward: parameters and host launch entry points.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include <cstdint>

namespace fa {

constexpr int kBwdTile = 128;  // keys per KV tile = query rows per Q tile

struct BwdParams {
    // preprocess inputs
    const float* o;         // [B, Hq, Lq, D] forward output
    const float* lse;       // [B, Hq, Lq] natural log
    const uint16_t* dout;   // bf16 [B, Hq, Lq, D]
    // outputs (fp32)
    float* dq;              // [B, Hq, Lq, D]  zeroed by the preprocess kernel, then accumulated
    float* dk;              // [B, Hkv, Lk, D]
    float* dv;              // [B, Hkv, Lk, D]
    // workspace, [B * Hq][Lq_pad] each
    float* delta;           // rowsum(O * dO); 0 on padding rows
    float* lse2;            // LSE * log2(e); +inf on rows without keys and on padding rows
    int B, Hq, Hkv, Lq, Lk, Lq_pad, group;
    int num_kv_tiles;       // ceil(Lk / 128)
    int num_q_tiles;        // ceil(Lq / 128)
    int num_items;          // B * Hkv * num_kv_tiles
    float scale;            // softmax_scale (multiplies dS)
    float scale_log2;       // softmax_scale * log2(e)
    int causal;
    int* err;
    int* diag;
    int fault;              // test hook: 1 = skip the first K/V load of every CTA
};

cudaError_t launch_bwd_pre(int D, const BwdParams& p, cudaStream_t stream);
cudaError_t launch_bwd(int D, bool causal, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& dout, const BwdParams& p, int grid, cudaStream_t stream);

}  // namespace fa
