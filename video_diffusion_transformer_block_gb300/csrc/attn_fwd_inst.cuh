// Launch helper for one attn_fwd_kernel instantiation.
#pragma once
#include "launch.h"

namespace vdtb {

template <int D, int BK, int MODE, int NQT, int NSTAGE>
cudaError_t launch_fwd_cfg(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                           cudaStream_t stream) {
  using Cfg = FwdCfg<D, BK, MODE, NQT, NSTAGE>;
  auto kernel = attn_fwd_kernel<D, BK, MODE, NQT, NSTAGE>;
  // the attribute is per device; setting it again is cheap and keeps multi-device use correct
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  // setmaxnreg.inc can only be granted what the launch allocated: refuse to
  // launch a build whose register count differs from the split the kernel assumes.
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, kernel);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != Cfg::kRegsLaunch) return cudaErrorInvalidDeviceFunction;
  long long grid = (long long)p.BH * p.n_qg * (MODE == kModeSplit ? p.n_split : 1);
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kernel<<<(unsigned)grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace vdtb
