// Kernel instances for head dimension 128.
#include "fa_fwd_kernel.cuh"
#include "fa_launch.h"

namespace fa {

template <int D, bool CAUSAL, bool VARLEN, int VAR>
cudaError_t launch_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const FwdParams& p, int grid, cudaStream_t stream)
{
    auto kern = fa_fwd_sm103_kernel<D, CAUSAL, VARLEN, VAR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FwdSmem<D, VAR>::kAlloc);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, FwdSmem<D, VAR>::kAlloc, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

#define FA_INSTANCE(D, C, V, VAR)                                                                        \
    template cudaError_t launch_fwd<D, C, V, VAR>(const CUtensorMap&, const CUtensorMap&,              \
                                                  const CUtensorMap&, const FwdParams&, int, cudaStream_t);

#if defined(FA_FP8)
// e4m3 inputs: D = 128, dense
FA_INSTANCE(128, false, false, kVarFp8)
FA_INSTANCE(128, true, false, kVarFp8)
#elif !defined(FA_VARIANTS)
#ifndef FA_HEAD_DIM
#define FA_HEAD_DIM 128
#endif
FA_INSTANCE(FA_HEAD_DIM, false, false, kVarNone)
FA_INSTANCE(FA_HEAD_DIM, true, false, kVarNone)
FA_INSTANCE(FA_HEAD_DIM, false, true, kVarNone)
FA_INSTANCE(FA_HEAD_DIM, true, true, kVarNone)
#else
// score variants: D = 128, dense and packed
FA_INSTANCE(128, false, false, kVarWindow)
FA_INSTANCE(128, false, true, kVarWindow)
FA_INSTANCE(128, false, false, kVarSoftcap)
FA_INSTANCE(128, false, true, kVarSoftcap)
FA_INSTANCE(128, false, false, kVarAlibi)
FA_INSTANCE(128, false, true, kVarAlibi)
#endif

}  // namespace fa
