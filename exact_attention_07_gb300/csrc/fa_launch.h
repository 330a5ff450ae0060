// Host-side launch entry points of the sm_103a kernels (one translation unit
// per head dimension instantiates them).
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include "fa_params.h"

namespace fa {


// D = query/key head dimension, DV = value head dimension.
template <int D, bool CAUSAL, bool VARLEN, int VAR = kVarNone, int DV = D>
cudaError_t launch_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const FwdParams& p, int grid, cudaStream_t stream);

// Builds the schedule of a variable-length batch into `sched`
// (see FwdParams::sched) and validates the offsets.  heads = Hq for the
// forward (bwd = 0; bwd = 2 counts paired-head tiles of 128 rows), Hkv for
// the backward (bwd = 1, which also writes the padded workspace row offsets).
cudaError_t launch_varlen_schedule(const int* cu_q, const int* cu_k, int num_seqs, int total_q,
                                   int total_k, int max_q, int max_k, int heads, int bwd, int* sched, int* err,
                                   cudaStream_t stream);

}  // namespace fa
