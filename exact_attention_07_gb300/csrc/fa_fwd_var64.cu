// Kernel instances of the score variants (key window, soft-capping, ALiBi),
// head dimension 64 (same source as the D = 128 unit).
#define FA_VARIANTS 1
#define FA_HEAD_DIM 64
#include "fa_fwd_d128.cu"
