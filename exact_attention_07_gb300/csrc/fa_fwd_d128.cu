// Kernel instances for head dimension 128.
#include "fa_fwd_kernel.cuh"
#include "fa_launch.h"

namespace fa {

template <int D, bool CAUSAL, bool VARLEN>
cudaError_t launch_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const FwdParams& p, int grid, cudaStream_t stream)
{
    auto kern = fa_fwd_sm103_kernel<D, CAUSAL, VARLEN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FwdSmem<D>::kAlloc);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, FwdSmem<D>::kAlloc, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

#define FA_INSTANCE(D, C, V)                                                                        \
    template cudaError_t launch_fwd<D, C, V>(const CUtensorMap&, const CUtensorMap&,              \
                                             const CUtensorMap&, const FwdParams&, int, cudaStream_t);

#ifndef FA_HEAD_DIM
#define FA_HEAD_DIM 128
#endif
FA_INSTANCE(FA_HEAD_DIM, false, false)
FA_INSTANCE(FA_HEAD_DIM, true, false)
FA_INSTANCE(FA_HEAD_DIM, false, true)
FA_INSTANCE(FA_HEAD_DIM, true, true)

}  // namespace fa
