// Kernel instances for head dimension 128.
#include "fa_fwd_kernel.cuh"
#include "fa_launch.h"

namespace fa {

template <int D, bool CAUSAL, bool VARLEN, int VAR, int DV>
cudaError_t launch_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const FwdParams& p, int grid, cudaStream_t stream)
{
    auto kern = fa_fwd_sm103_kernel<D, CAUSAL, VARLEN, VAR, DV>;
    constexpr int kSmem = fwd_smem_alloc<D, VARLEN, VAR, DV>();
    cudaError_t e = smem_limit_once<fa_fwd_sm103_kernel<D, CAUSAL, VARLEN, VAR, DV>>(kSmem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, kSmem, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

#define FA_INSTANCE_DV(D, C, V, VAR, DV)                                                                 \
    template cudaError_t launch_fwd<D, C, V, VAR, DV>(const CUtensorMap&, const CUtensorMap&,          \
                                                      const CUtensorMap&, const FwdParams&, int, cudaStream_t);
#define FA_INSTANCE(D, C, V, VAR) FA_INSTANCE_DV(D, C, V, VAR, D)

#if defined(FA_D192)
// query/key head dimension 192, value head dimension 128
FA_INSTANCE_DV(192, false, false, kVarNone, 128)
FA_INSTANCE_DV(192, true, false, kVarNone, 128)
FA_INSTANCE_DV(192, false, true, kVarNone, 128)
FA_INSTANCE_DV(192, true, true, kVarNone, 128)
#elif defined(FA_FP8)
// e4m3 inputs: D = 128, dense
FA_INSTANCE(128, false, false, kVarFp8)
FA_INSTANCE(128, true, false, kVarFp8)
#else
#ifndef FA_HEAD_DIM
#define FA_HEAD_DIM 128
#endif
#if !defined(FA_VARIANTS)
FA_INSTANCE(FA_HEAD_DIM, false, false, kVarNone)
FA_INSTANCE(FA_HEAD_DIM, true, false, kVarNone)
FA_INSTANCE(FA_HEAD_DIM, false, true, kVarNone)
FA_INSTANCE(FA_HEAD_DIM, true, true, kVarNone)
#else
// score variants, dense and packed
FA_INSTANCE(FA_HEAD_DIM, false, false, kVarWindow)
FA_INSTANCE(FA_HEAD_DIM, false, true, kVarWindow)
FA_INSTANCE(FA_HEAD_DIM, false, false, kVarSoftcap)
FA_INSTANCE(FA_HEAD_DIM, false, true, kVarSoftcap)
FA_INSTANCE(FA_HEAD_DIM, false, false, kVarAlibi)
FA_INSTANCE(FA_HEAD_DIM, false, true, kVarAlibi)
FA_INSTANCE(FA_HEAD_DIM, false, false, kVarCapAlibi)
FA_INSTANCE(FA_HEAD_DIM, false, true, kVarCapAlibi)
#endif
#endif

}  // namespace fa
