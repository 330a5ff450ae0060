// Kernel instances for query/key head dimension 192 with value head dimension
// 128 (same source as the D = 128 unit).
#define FA_D192 1
#include "fa_fwd_d128.cu"
