"""CPU oracle for stabilised BF16 flash attention (forward and backward).

TEST INFRASTRUCTURE, not part of the product. Only ``tests/``,
``__graft_entry__.smoke()``, and ``bench.py``'s CPU-baseline leg and its
``--impl reference`` arm (both time the oracle on the host cores) may
import, call or execute anything in this package. The CUDA path never imports
it and it never imports the CUDA path; the two share no code, header, helper,
table or constant. The only shared module is the seeded input generator
(``precision_flash_attention_gb300.inputs``), which holds none of the method's
arithmetic and which this package does not import either.

The oracle is the plain, whole-row definition written with numpy in float64,
plus a BF16-emulation mode with the cast points of a fused kernel (see
``oracle.attention``). Its pins (tests marked ``not gpu``) tie it to what the
pages and mathematics fix: the two worked BF16 traces, a library softmax
reference, closed forms for N = 1 and causal row 0, shift invariance across
the three fix modes, the delta identity, central finite differences of the
backward pass, and brute-force counts on integer-valued inputs.
"""
from .attention import (EPS_SHIFT, TIE_BINS, attn_bwd, attn_bwd_rows, attn_delta, attn_delta_alt, attn_fwd,
                        attn_fwd_blockwise, attn_fwd_head, attn_fwd_monitor, attn_fwd_unfused, fix_shift, scores,
                        visible)
from .bf16 import (BF16_ONE_THRESHOLD, E2M1_MAX, E4M3_MAX, MX_BLOCK, bf16_rne, bf16_sum, e2m1_rne,
                   e4m3_rne, fp32, ftz32, mx_e2m1)

__all__ = [
    "EPS_SHIFT", "TIE_BINS", "attn_bwd", "attn_bwd_rows", "attn_fwd_monitor", "attn_fwd_unfused", "attn_fwd_blockwise", "attn_delta", "attn_delta_alt", "attn_fwd", "attn_fwd_head",
    "fix_shift", "scores", "visible", "BF16_ONE_THRESHOLD", "bf16_rne", "bf16_sum", "fp32",
    "ftz32", "E2M1_MAX", "E4M3_MAX", "MX_BLOCK", "e2m1_rne", "e4m3_rne", "mx_e2m1",
]
