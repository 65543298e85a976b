"""Algorithmic HBM bytes of the calls: what the method must move, no more.

"feat(kda): add packed-input CuTe decode kernel" (PR #4417), section "DRAM
utilization": per step the decode reads and rewrites the whole bf16 state of
each row (12 x 128 x 128 values, a 786 KB round trip) plus about 15 KB of
activations. The same count is used here, per row:

  T=1 decode, active row:  state read + write 2*H*V*K*2
                           + q, k, v, g_raw 4*H*128*2 + beta H*2 + out H*V*2 + index 4
  inactive row:            index 4 + out H*V*2 (the kernel writes zeros)
  T-token verify:          the state once each way + T x (activations + outputs)
  ring verify (h live entries, fold f in {0, 1}):
                           checkpoint read H*V*K*2 + (h + T) ring entries of
                           k~ (bf16), u~ (bf16), G (fp32) per head
                           + T x (activations + outputs) + index + hist_len
                           + f x checkpoint write
  per call:                A_log H*4 + dt_bias H*128*4
  T=1 decode on an fp8 pool (kda_fp8.h), active row:
                           codes read + write 2*H*V*K + row scales 2*H*V*4
                           + the same activations, output and index; the
                           T-token verify and the ring verify on an fp8 pool
                           count their checkpoint as codes + scales likewise
  varlen prefill (kda_prefill.h), an active sequence of n tokens:
                           its slot once each way + n x (activations + outputs)
                           + index + two cu_seqlens entries. The prefill is
                           bound by arithmetic, not bytes: per token and head
                           the step does 7 flops per state element (decay 1,
                           two dot products 4, update 2), 7*K*V in all.
"""

H, K, V = 12, 128, 128

STATE_BYTES = H * V * K * 2                  # one row's state, one direction: 393,216
TOKEN_IO_BYTES = 4 * H * K * 2 + H * 2 + H * V * 2  # q, k, v, g_raw, beta, out: 15,384
RING_ENTRY_BYTES = H * (K * 2 + V * 2 + K * 4)      # k~, u~, G for all heads: 12,288
INDEX_BYTES = 4
PER_CALL_BYTES = H * 4 + H * K * 4           # A_log, dt_bias: 6,192
FP8_STATE_BYTES = H * V * K + H * V * 4      # codes and row scales, one direction: 202,752


def decode_bytes(n_active, n_inactive=0):
    return (n_active * (2 * STATE_BYTES + TOKEN_IO_BYTES + INDEX_BYTES)
            + n_inactive * (INDEX_BYTES + H * V * 2) + PER_CALL_BYTES)


def verify_bytes(n_active, T, n_inactive=0):
    return (n_active * (2 * STATE_BYTES + T * TOKEN_IO_BYTES + INDEX_BYTES)
            + n_inactive * (INDEX_BYTES + T * H * V * 2) + PER_CALL_BYTES)


def ring_row_bytes(h, T, fold, state_bytes=STATE_BYTES):
    return (state_bytes + (h + T) * RING_ENTRY_BYTES + T * TOKEN_IO_BYTES + INDEX_BYTES + 4
            + (state_bytes if fold else 0))


def ring_bytes(hists, T, flush_min, n_inactive=0, state_bytes=STATE_BYTES):
    """hists: hist_len of each active row before the call; state_bytes: one
    checkpoint, one direction (FP8_STATE_BYTES for an fp8 pool)."""
    return (sum(ring_row_bytes(h, T, h >= flush_min, state_bytes) for h in hists)
            + n_inactive * (INDEX_BYTES + T * H * V * 2) + PER_CALL_BYTES)


def decode_fp8_bytes(n_active, n_inactive=0):
    return (n_active * (2 * FP8_STATE_BYTES + TOKEN_IO_BYTES + INDEX_BYTES)
            + n_inactive * (INDEX_BYTES + H * V * 2) + PER_CALL_BYTES)


def verify_fp8_bytes(n_active, T, n_inactive=0):
    return (n_active * (2 * FP8_STATE_BYTES + T * TOKEN_IO_BYTES + INDEX_BYTES)
            + n_inactive * (INDEX_BYTES + T * H * V * 2) + PER_CALL_BYTES)


def prefill_bytes(lengths, n_inactive_tokens=0):
    """Active sequences of the given lengths, plus inactive tokens (zero outputs)."""
    return (sum(2 * STATE_BYTES + n * TOKEN_IO_BYTES + INDEX_BYTES + 8 for n in lengths)
            + n_inactive_tokens * H * V * 2 + PER_CALL_BYTES)


def prefill_flops(tokens, heads=H):
    """Arithmetic of the recurrence over `tokens` active tokens of `heads` heads."""
    return tokens * heads * 7 * K * V
