// Launch parameters shared by the host launcher and the sm_103a kernels.
#pragma once

#include <cstdint>

namespace fa {

struct FwdParams {
    float* o;          // fp32 output
    float* lse;        // fp32 output, natural log
    int B, Hq, Hkv;    // batch (dense only), query heads, KV heads
    int Lq, Lk;        // dense sequence lengths (unused for varlen)
    int group;         // Hq / Hkv
    float scale_log2;  // softmax_scale * log2(e)
    int heads_per_section;  // KV heads per L2-sized scheduling section
    int num_tiles;          // dense: number of work tiles
    // variable-length batches
    const int* cu_q;
    const int* cu_k;
    const int* sched;  // [0] tiles, [1..n+1] tile prefix in schedule order, [n+2..2n+1] order
    int num_seqs;
    int total_q;
    // programmable variants (kernels instantiated with VAR > 0)
    int win_left, win_right;  // key window around the query's aligned position; < 0 = unlimited
    float cap_in;             // soft-capping: scale / cap
    float cap_out;            // soft-capping: cap * log2(e)
    const float* alibi;       // ALiBi: per query head slope (natural-log units)
    // error reporting
    int* err;
    int* diag;
    int fault;  // test hook: 1 = the producer drops the first K tile of each CTA
};

// Rows of one Q tile and keys of one KV tile; a CTA owns two Q tiles.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kRowsPerCta = 2 * kBlockM;
constexpr int kThreads = 512;

// Score variants of the forward kernel (FlashAttention from Scratch, sec. 12):
// 0 = plain, 1 = key window, 2 = key window + soft-capping, 3 = key window + ALiBi.
enum : int { kVarNone = 0, kVarWindow = 1, kVarSoftcap = 2, kVarAlibi = 3 };

}  // namespace fa
