"""CPU oracle for the KDA (Kimi Delta Attention) gated delta-rule decode step.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import, call or execute anything in this
package. The product path (``linear_attention_ssm_step_gb300``) never does:
it runs the CUDA library or fails.

The oracle is plain numpy in fp64. It rounds to bf16 (and to fp32 for the
ring's cumulative log-decay) exactly where the method stores values, with a
direct fp64 -> bf16 round-to-nearest-even that never passes through fp32.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
(the fp8 state pool in ``tests/test_oracle_pins_fp8.py``, the varlen prefill in
``tests/test_oracle_pins_prefill.py``)
against closed forms, invariants, brute force at K=V=4 and library rounding
routines. No function is "parity unpinned".
"""

from .kda_oracle import (  # noqa: F401
    round_to_bf16,
    round_to_fp32,
    l2_normalize,
    gate_log_decay,
    beta_from_logit,
    prologue,
    decode_step_math,
    kda_decode,
    kda_verify,
    ring_replay,
    ring_fold_closed_form,
    kda_verify_ring,
    RING_ERR_HIST_LEN,
    RING_ERR_CACHE_BASE,
    L2_EPS,
    GATE_RAW,
    GATE_PRECOMPUTED,
)
from .kda_fp8_oracle import (  # noqa: F401,E402
    e4m3_decode,
    e4m3_encode,
    row_exponent,
    requantize_rows,
    dequantize,
    kda_decode_fp8,
    kda_verify_ring_fp8,
)
from .kda_prefill_oracle import (  # noqa: F401,E402
    kda_prefill,
    PREFILL_ERR_SEQLENS,
)
