// Backward kernel instances of the score variants (key window, soft-capping,
// ALiBi), head dimension 128 (same source as the main backward unit).
#define FA_BWD_VARIANTS 1
#include "fa_bwd.cu"
