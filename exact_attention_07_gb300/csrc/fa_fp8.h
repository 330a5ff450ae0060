// FP8 forward: input preparation (incoherent processing + block quantisation).
#pragma once

#include <cuda_runtime_api.h>

#include <cstdint>

namespace fa {

constexpr int kFp8Tile = 128;  // rows per quantisation tile (= the kernel's Q and KV tiles)

struct Fp8PrepParams {
    const uint16_t* q;   // bf16 [B*Hq][Lq][128]
    const uint16_t* k;   // bf16 [B*Hkv][Lk][128]
    const uint16_t* v;   // bf16 [B*Hkv][Lk][128]
    const float* signs;  // [128] +-1 (the random signs of the rotation)
    uint8_t* qc;         // e4m3 [B*Hq][Lq][128]   codes of Q diag(signs) H / sqrt(128)
    uint8_t* kc;         // e4m3 [B*Hkv][Lk][128]  codes of K diag(signs) H / sqrt(128)
    uint8_t* vt;         // e4m3 [B*Hkv][128][Lk_pad] codes of V, transposed (zero beyond Lk)
    float* sq;           // [B*Hq][nq]   scale of each 128-row Q tile
    float* sk;           // [B*Hkv][nk]  scale of each 128-row K tile
    float* sv;           // [B*Hkv]      scale of each V slice
    unsigned* vmax;      // [B*Hkv]      scratch: amax of V slices (float bits)
    int B, Hq, Hkv, Lq, Lk, Lk_pad, nq, nk;
};

// Runs the three preparation kernels (Q/K rotation and quantisation, V
// amax, V quantisation and transpose) on `stream`; vmax must be zeroed first.
cudaError_t launch_fp8_prepare(const Fp8PrepParams& p, cudaStream_t stream);

}  // namespace fa
