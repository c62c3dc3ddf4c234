// The fused forward path at d = 128 with the two CTAs of a cluster paired on
// every product (tcgen05 cta_group::2, M = 256): the attention forward kernel of
// attn_fwd.cuh with PAIR set, for the three shift modes, causal or not, with or
// without the diagnostic counters.
#define PFA_FWD_NO_TRACE
#include "attn_fwd.cuh"

namespace pfa {
namespace {

template <int MODE>
cudaError_t dispatch_causal(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& a, cudaStream_t st) {
  const bool count = a.counters != nullptr;
  if (a.s.causal)
    return count ? fwd::launch_fwd_pair_t<MODE, true, 1>(tq, tk, tv, a, st)
                 : fwd::launch_fwd_pair_t<MODE, true, 0>(tq, tk, tv, a, st);
  return count ? fwd::launch_fwd_pair_t<MODE, false, 1>(tq, tk, tv, a, st)
               : fwd::launch_fwd_pair_t<MODE, false, 0>(tq, tk, tv, a, st);
}

}  // namespace

cudaError_t launch_fwd_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& a, cudaStream_t stream) {
  switch (a.fix_mode) {
    case 0: return dispatch_causal<0>(tq, tk, tv, a, stream);
    case 1: return dispatch_causal<1>(tq, tk, tv, a, stream);
    default: return dispatch_causal<2>(tq, tk, tv, a, stream);
  }
}

}  // namespace pfa
