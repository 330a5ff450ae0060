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
    // 1: a work tile is two query heads of one KV head over the same 128 rows
    // (causal, even GQA groups); 0: one query head over 256 rows
    int pair_heads;
    // key windows: 1 = row blocks from the last (when later blocks see at
    // least as many keys, so that the longest tiles come first), 0 = from the first
    int desc_tiles;
    // variable-length batches
    const int* cu_q;
    const int* cu_k;
    // Precomputed schedule ([0] tiles, [1..n+1] tile prefix in schedule order,
    // [n+2..2n+1] order, n = num_seqs), or null: then every CTA builds the
    // schedule of sequences [seq_begin, seq_begin + seq_count) in its own
    // shared memory (at most varlen_sched_max_seqs(D, DV) of them).
    const int* sched;
    int num_seqs;      // sequences in the whole batch
    int seq_begin, seq_count;
    int total_q, total_k;
    int max_q, max_k;  // the caller's length bounds, checked per sequence
    // programmable variants (kernels instantiated with VAR > 0)
    int win_left, win_right;  // key window around the query's aligned position; < 0 = unlimited
    float cap_in;             // soft-capping: scale / cap
    float cap_out;            // soft-capping: cap * log2(e)
    const float* alibi;       // ALiBi: per query head slope (natural-log units)
    // FP8 forward (VAR = kVarFp8): dequantisation scales of the e4m3 inputs
    const float* fp8_sq;      // [B*Hq][fp8_nq] per 128-row Q tile
    const float* fp8_sk;      // [B*Hkv][fp8_nk] per 128-key K tile
    const float* fp8_sv;      // [B*Hkv] per V slice
    int fp8_nq, fp8_nk;
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

// Variants of the forward kernel: 0 = plain, 1 = key window, 2 = key window +
// soft-capping, 3 = key window + ALiBi (FlashAttention from Scratch, sec. 12),
// 4 = e4m3 inputs with per-tile scales (sec. 10.3), 5 = key window +
// soft-capping followed by ALiBi.
enum : int { kVarNone = 0, kVarWindow = 1, kVarSoftcap = 2, kVarAlibi = 3, kVarFp8 = 4, kVarCapAlibi = 5 };
constexpr bool var_softcap(int v) { return v == kVarSoftcap || v == kVarCapAlibi; }
constexpr bool var_alibi(int v) { return v == kVarAlibi || v == kVarCapAlibi; }

// Sequences one launch of a packed batch can schedule in shared memory
// (what the forward kernel's layout leaves free at each head dimension); the
// host splits larger batches into launches of at most this many sequences.
constexpr int varlen_sched_max_seqs(int D, int DV) { return D == DV ? 1536 : 64; }
constexpr bool var_window(int v) { return v == kVarWindow || var_softcap(v) || var_alibi(v); }

}  // namespace fa
