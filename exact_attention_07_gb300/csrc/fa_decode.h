// Split-KV decode forward: parameters and host launch entry points.
//
// Decode has few query rows per KV head (one new token, or a handful under
// speculative decoding) and a long key range.  Query-tile parallelism is gone,
// so the key range of each (batch, KV head) is split into independent
// partitions that run as separate CTAs, and a second kernel combines their
// partial results by their log-sum-exp weights (FlashAttention from Scratch,
// sec. 9.1 "Split the long dimension that remains" and sec. 4.3 "Merge
// independently computed partitions").
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include <cstddef>
#include <cstdint>

namespace fa {

constexpr int kDecThreads = 256;  // threads of one partial CTA
constexpr int kDecKeys = 64;      // keys per K/V tile
constexpr int kDecMaxRows = 16;   // query rows sharing one KV head: (Hq / Hkv) * Lq

struct DecodeParams {
    const uint16_t* q;  // bf16 [B, Hq, Lq, D]
    float* o;           // [B, Hq, Lq, D]
    float* lse;         // [B, Hq, Lq], natural log
    float* o_part;      // [B * Hkv, num_splits, R, D]  normalised partial outputs
    float* l_part;      // [B * Hkv, num_splits, R]     partial log-sum-exp, base 2
    int B, Hq, Hkv, Lq, Lk, group;
    int R;                // group * Lq query rows per KV head
    int num_splits;       // partitions of the key range per (batch, KV head)
    int tiles_per_split;  // key tiles of one partition (the last may have fewer)
    int num_tiles;        // ceil(Lk / keys per tile): 64 keys (FP32 pipes), 16384 / D (tensor cores)
    int causal;
    float scale_log2;  // softmax_scale * log2(e)
    int* err;
    int* diag;
    int fault;  // test hook: 1 = skip the first tile load of every CTA
};

// Rows handled per lane group in the P.V phase: the kernel is instantiated for
// rows_per_thread in {1, 2, 4, 8} and R <= (256 / D) * rows_per_thread.
int decode_rows_per_thread(int D, int R);

// CTAs of the partial kernel that fit on one SM (occupancy calculator).
int decode_ctas_per_sm(int D, int rows_per_thread);

cudaError_t launch_decode_partial(int D, int rows_per_thread, const CUtensorMap& k, const CUtensorMap& v,
                                  const DecodeParams& p, int grid, cudaStream_t stream);

cudaError_t launch_decode_merge(int D, const DecodeParams& p, cudaStream_t stream);

// Tensor-core partials (D = 64 or 128, 2 <= R <= 16): tiles of 16384 / D keys
// (32 KB of K or of V), loaded as [128 keys][64 dimensions] boxes, one
// persistent CTA per SM (grid <= SM count) walking the (batch, KV head,
// partition) items.
constexpr int kDecTcKeys = 128;  // keys of one TMA box
constexpr int decode_tc_keys(int D) { return 16384 / D; }
cudaError_t launch_decode_tc(int D, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                             const DecodeParams& p, int grid, cudaStream_t stream);

}  // namespace fa
