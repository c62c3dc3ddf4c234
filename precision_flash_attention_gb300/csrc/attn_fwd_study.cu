// The forward kernel's study variants (attn_fwd.cuh): the monitor (the
// operational count of BF16 Pbar == 1 handed to the Pbar V product, and the
// histogram of tie multiplicities) and the unfused profile, which rounds each key
// tile's product Pbar V to BF16 and accumulates it across tiles in BF16 -- the
// way an implementation that stores the unnormalised product in BF16 computes O
// (priors.kr post "BF16 플래시 어텐션은 왜 수천 스텝 뒤에 무너질까", caveats:
// the analysed code is FlashAttention 2 as PyTorch operations that keep P V in
// BF16).
#define PFA_FWD_NO_TRACE
#include "attn_fwd.cuh"

namespace pfa {
namespace {

// MON = 2 counts everything the monitor and the counters report (either output
// may be absent); the profile without either counts nothing.
template <int D, int MODE, bool PROFILE>
cudaError_t dispatch_causal(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdArgs& a, cudaStream_t st) {
  const bool count = a.counters != nullptr || a.monitor != nullptr;
  if (a.s.causal)
    return count ? fwd::launch_fwd_t<D, MODE, true, 2, PROFILE>(tq, tk, tv, a, st)
                 : fwd::launch_fwd_t<D, MODE, true, 0, PROFILE>(tq, tk, tv, a, st);
  return count ? fwd::launch_fwd_t<D, MODE, false, 2, PROFILE>(tq, tk, tv, a, st)
               : fwd::launch_fwd_t<D, MODE, false, 0, PROFILE>(tq, tk, tv, a, st);
}

template <int D, bool PROFILE>
cudaError_t dispatch_mode(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdArgs& a, cudaStream_t st) {
  switch (a.fix_mode) {
    case 0: return dispatch_causal<D, 0, PROFILE>(tq, tk, tv, a, st);
    case 1: return dispatch_causal<D, 1, PROFILE>(tq, tk, tv, a, st);
    default: return dispatch_causal<D, 2, PROFILE>(tq, tk, tv, a, st);
  }
}

}  // namespace

cudaError_t launch_fwd_study(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FwdArgs& a, cudaStream_t stream) {
  if (a.profile) return dispatch_mode<64, true>(tq, tk, tv, a, stream);
  if (a.s.d == 64) return dispatch_mode<64, false>(tq, tk, tv, a, stream);
  return dispatch_mode<128, false>(tq, tk, tv, a, stream);
}

}  // namespace pfa
