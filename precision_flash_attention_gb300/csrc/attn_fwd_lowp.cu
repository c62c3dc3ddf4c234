// The forward kernel (attn_fwd.cuh) with the Pbar operand rounded to a narrower
// format than BF16: FP8 E4M3, or MXFP4 (E2M1 with one power-of-two scale per 32
// keys). A study of the question the priors.kr post "BF16 플래시 어텐션은 왜 수천
// 스텝 뒤에 무너질까" leaves open (open questions): how the rounding that makes
// Pbar exactly 1 behaves with fewer mantissa bits. d = 64, with the monitor (the
// operational count of Pbar == 1 handed to the product), fused (FP32 Obar) or
// with the unfused BF16 profile.
#define PFA_FWD_NO_TRACE
#include "attn_fwd.cuh"

namespace pfa {
namespace {

template <int MODE, bool PROFILE, int PBAR>
cudaError_t dispatch_causal(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& a, cudaStream_t st) {
  if (a.s.causal) return fwd::launch_fwd_t<64, MODE, true, 2, PROFILE, PBAR>(tq, tk, tv, a, st);
  return fwd::launch_fwd_t<64, MODE, false, 2, PROFILE, PBAR>(tq, tk, tv, a, st);
}

template <bool PROFILE, int PBAR>
cudaError_t dispatch_mode(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdArgs& a, cudaStream_t st) {
  switch (a.fix_mode) {
    case 0: return dispatch_causal<0, PROFILE, PBAR>(tq, tk, tv, a, st);
    case 1: return dispatch_causal<1, PROFILE, PBAR>(tq, tk, tv, a, st);
    default: return dispatch_causal<2, PROFILE, PBAR>(tq, tk, tv, a, st);
  }
}

template <int PBAR>
cudaError_t dispatch_profile(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FwdArgs& a, cudaStream_t st) {
  return a.profile ? dispatch_mode<true, PBAR>(tq, tk, tv, a, st)
                   : dispatch_mode<false, PBAR>(tq, tk, tv, a, st);
}

}  // namespace

cudaError_t launch_fwd_lowp(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& a, cudaStream_t stream) {
  if (a.pbar == fwd::kPbarE4m3) return dispatch_profile<fwd::kPbarE4m3>(tq, tk, tv, a, stream);
  return dispatch_profile<fwd::kPbarMxfp4>(tq, tk, tv, a, stream);
}

}  // namespace pfa
