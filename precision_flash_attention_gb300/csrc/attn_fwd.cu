// The fused forward path: the attention forward kernel (attn_fwd.cuh) with the
// FP32 Obar accumulator, instantiated for d = 64 and 128, the three shift modes,
// causal or not, with or without the diagnostic counters.
#include "attn_fwd.cuh"

namespace pfa {
namespace {

template <int D, int MODE>
cudaError_t dispatch_causal(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& a, cudaStream_t st) {
  const bool count = a.counters != nullptr;
  if (a.s.causal)
    return count ? fwd::launch_fwd_t<D, MODE, true, 1, false>(tq, tk, tv, a, st)
                 : fwd::launch_fwd_t<D, MODE, true, 0, false>(tq, tk, tv, a, st);
  return count ? fwd::launch_fwd_t<D, MODE, false, 1, false>(tq, tk, tv, a, st)
               : fwd::launch_fwd_t<D, MODE, false, 0, false>(tq, tk, tv, a, st);
}

template <int D>
cudaError_t dispatch_mode(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdArgs& a, cudaStream_t st) {
  switch (a.fix_mode) {
    case 0: return dispatch_causal<D, 0>(tq, tk, tv, a, st);
    case 1: return dispatch_causal<D, 1>(tq, tk, tv, a, st);
    default: return dispatch_causal<D, 2>(tq, tk, tv, a, st);
  }
}

}  // namespace

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& a, cudaStream_t stream) {
  if (a.s.d == 64) return dispatch_mode<64>(tq, tk, tv, a, stream);
  return dispatch_mode<128>(tq, tk, tv, a, stream);
}

}  // namespace pfa
