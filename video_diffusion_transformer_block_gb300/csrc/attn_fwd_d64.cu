// attn_fwd_kernel and attn_na_persist_kernel instantiations for head dim 64.
#include "attn_fwd_inst.cuh"

namespace vdtb {

cudaError_t launch_attn_fwd_d64(int BK, int mode, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const FwdParams& p, cudaStream_t stream) {
  if (mode == kModeDense && BK == 128) return launch_fwd_cfg<64, 128, kModeDense, 2, 4>(tq, tk, tv, p, stream);
  if (mode == kModeSparse && BK == 128) return launch_fwd_cfg<64, 128, kModeSparse, 2, 4>(tq, tk, tv, p, stream);
  if (mode == kModeSparse && BK == 64) return launch_fwd_cfg<64, 64, kModeSparse, 2, 4>(tq, tk, tv, p, stream);
  if (mode == kModeSplit && BK == 128) return launch_fwd_cfg<64, 128, kModeSplit, 1, 4>(tq, tk, tv, p, stream);
  if (mode == kModeSparseFused && BK == 128) return launch_fwd_cfg<64, 128, kModeSparseFused, 2, 6>(tq, tk, tv, p, stream);
  if (mode == kModeSparseFused && BK == 64) return launch_fwd_cfg<64, 64, kModeSparseFused, 2, 8>(tq, tk, tv, p, stream);
  if (mode == kModeNA1x8x16 && BK == 128 && p.na_pair_axis == 3) return launch_fwd_cfg<64, 128, kModeNA1x8x16, 1, 4>(tq, tk, tv, p, stream);
  if (mode == kModeNA2x8x8 && BK == 128 && p.na_pair_axis == 3) return launch_fwd_cfg<64, 128, kModeNA2x8x8, 1, 4>(tq, tk, tv, p, stream);
  if (mode == kModeNA4x4x8 && BK == 128 && p.na_pair_axis == 3) return launch_fwd_cfg<64, 128, kModeNA4x4x8, 1, 4>(tq, tk, tv, p, stream);
  if (mode == kModeNA1x8x16 && BK == 128) return launch_fwd_cfg<64, 128, kModeNA1x8x16, 2, 6>(tq, tk, tv, p, stream);
  if (mode == kModeNA2x8x8 && BK == 128) return launch_fwd_cfg<64, 128, kModeNA2x8x8, 2, 6>(tq, tk, tv, p, stream);
  if (mode == kModeNA4x4x8 && BK == 128) return launch_fwd_cfg<64, 128, kModeNA4x4x8, 2, 6>(tq, tk, tv, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_na_persist_d64(int mode, int keys, const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const FwdParams& p, cudaStream_t stream) {
  if (keys == kNAKeysWide)
    return mode == kModeNA4x4x8 ? launch_na_persist_cfg<64, kModeNA4x4x8, kNAKeysWide>(tq, tk, tv, p, stream)
                                : cudaErrorInvalidValue;
  if (keys == kNAKeysWideF8)
    return mode == kModeNA4x4x8 ? launch_na_persist_cfg<64, kModeNA4x4x8, kNAKeysWideF8>(tq, tk, tv, p, stream)
                                : cudaErrorInvalidValue;
  if (mode == kModeNA1x8x16) return launch_na_persist_cfg<64, kModeNA1x8x16, kNAKeysBrick>(tq, tk, tv, p, stream);
  if (mode == kModeNA2x8x8) return launch_na_persist_cfg<64, kModeNA2x8x8, kNAKeysBrick>(tq, tk, tv, p, stream);
  if (mode == kModeNA4x4x8) return launch_na_persist_cfg<64, kModeNA4x4x8, kNAKeysBrick>(tq, tk, tv, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace vdtb
