// Kernel instances of the FP8 forward (e4m3 inputs with per-tile scales),
// head dimension 128 (same source as the D = 128 unit).
#define FA_FP8 1
#include "fa_fwd_d128.cu"
