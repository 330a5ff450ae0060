// Backward kernel instances of the score variants (key window, soft-capping,
// ALiBi), head dimension 64 (same source as the main backward unit).
#define FA_BWD_VARIANTS 1
#define FA_BWD_HEAD_DIM 64
#include "fa_bwd.cu"
