// Launch helper for one attn_fwd_kernel instantiation.
#pragma once
#include "launch.h"
#include "na_persist.cuh"

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

// The persistent neighbourhood kernel: one CTA per SM (fewer when there are
// fewer than two bricks per SM), each of its two tiles walking its own bricks.
template <int D, int MODE, int KEYS>
cudaError_t launch_na_persist_cfg(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const FwdParams& p, cudaStream_t stream) {
  using Cfg = NAPersistCfg<D, MODE, KEYS>;
  auto kernel = attn_na_persist_kernel<D, MODE, KEYS>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, kernel);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != Cfg::kRegsLaunch) return cudaErrorInvalidDeviceFunction;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long units = (long long)p.BH * p.na_nq[0] * p.na_nq[1] * p.na_nq[2];
  if (units <= 0 || units > 0x7fffffffLL || sms <= 0) return cudaErrorInvalidConfiguration;
  const long long grid = (units + 1) / 2 < sms ? (units + 1) / 2 : sms;
  kernel<<<(unsigned)grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace vdtb
