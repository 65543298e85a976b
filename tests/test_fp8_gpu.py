"""kda_decode_fp8 (T = 1 on an fp8 E4M3 state pool) on the GPU against the fp64
oracle of the library's fp8 reading, through the C ABI.

What is compared, and why so:
  * outputs: the decode's tolerance, 2e-2 + 2e-2 |o_ref| (they come from the
    unrounded new state, as in the bf16 decode);
  * the new state: both sides decide the requantization in fp32, but the
    kernel's fp32 new state and the oracle's fp64 one rounded to fp32 differ
    by fp32 rounding (the terms of a row are of the size M of its largest
    element, so by up to a few 2^-24 M). A code, or a row's exponent, can
    therefore fall on the other side of a rounding boundary. What is unique
    is checked everywhere: the GPU's dequantized row lies within half an E4M3
    step (at the GPU's own row scale) plus 2^-18 M of the oracle's unrounded
    new state; and the codes and exponents equal the oracle's except for a
    small fraction (at most 1e-3 of the codes, 1e-3 of the rows), each such
    exponent one away and each such code one step away;
  * inactive rows and untouched slots: bit for bit (zero output, codes and
    scales unchanged).
"""

import numpy as np
import pytest
import torch

import oracle
from harness import assert_output_close, f64
from linear_attention_ssm_step_gb300 import kda, workloads

pytestmark = pytest.mark.gpu

LB = -5.0


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def make(B, N, seed, layout="separate", inactive_frac=0.0, H=12):
    w = workloads.decode_inputs(B, N, seed=seed, layout=layout, inactive_frac=inactive_frac, H=H)
    codes, scales = workloads.fp8_pool(N, H=H, seed=seed + 7)
    return w, codes, scales


def gpu_call(wd, codes, scales, **kw):
    return kda.kda_decode_fp8(codes, scales, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit,
                              wd.A_log, wd.dt_bias, lower_bound=LB, **kw)


def oracle_call(w, codes, scales, rows=None, scale=1.0):
    sub = w if rows is None else w.select_rows(rows)
    return oracle.kda_decode_fp8(codes.numpy(), scales.double().numpy(), sub.state_indices.numpy(), f64(sub.q),
                                 f64(sub.k), f64(sub.v), f64(sub.g_raw), f64(sub.beta_logit), f64(sub.A_log),
                                 f64(sub.dt_bias), LB, scale)


def check_state(got_codes, got_scales, ref_codes, ref_scales, S_new, slack=2.0 ** -18):
    """The new state of the active slots: got/ref codes [nA, H, V, K] uint8,
    scales [nA, H, V]; S_new the oracle's unrounded new state; slack the
    kernel's own error before the rounding, as a fraction of the row's
    largest magnitude."""
    got_e = np.log2(got_scales).astype(np.int64)
    ref_e = np.log2(ref_scales).astype(np.int64)
    assert np.array_equal(np.ldexp(1.0, got_e), got_scales), "scales must be powers of two"
    row_diff = got_e != ref_e
    assert np.all(np.abs(got_e - ref_e) <= 1)
    assert row_diff.mean() <= 1e-3, f"{row_diff.sum()} of {row_diff.size} row exponents differ"
    deq = oracle.dequantize(got_codes, got_scales)
    M = np.max(np.abs(S_new), axis=-1, keepdims=True)
    ax = np.maximum(np.abs(S_new), 1e-300)
    qexp = np.maximum(np.floor(np.log2(ax)) - 3, got_e[..., None] - 9).astype(np.int64)
    bound = np.ldexp(0.5, qexp) + slack * M
    excess = np.abs(deq - S_new) / bound
    assert excess.max() <= 1.0, f"dequantized state off by {excess.max():.3f} x the bound"
    same_row = ~row_diff[..., None]
    code_diff = (got_codes != ref_codes) & same_row & ((got_codes | ref_codes) & 0x7F != 0)
    assert code_diff.mean() <= 1e-3, f"{code_diff.sum()} codes differ"
    if code_diff.any():
        step = np.abs(oracle.e4m3_decode(got_codes[code_diff]) - oracle.e4m3_decode(ref_codes[code_diff]))
        ref_mag = np.abs(oracle.e4m3_decode(ref_codes[code_diff]))
        # at most two code steps: 2^(E-3) each in the binade [2^E, 2^(E+1)), and
        # the subnormal quantum 2^-9 = the step of the smallest normal binade 2^-6
        assert np.all(step <= np.ldexp(1.0, (np.floor(np.log2(np.maximum(ref_mag, 2.0 ** -6))) - 2).astype(int)))


def run_and_check(w, codes, scales, dev, scale=1.0, **kw):
    wd = w.to(dev)
    c_d, s_d = codes.to(dev), scales.to(dev)
    out = gpu_call(wd, c_d, s_d, scale=scale, **kw)
    torch.cuda.synchronize()
    ref_c, ref_s, ref_out, info = oracle_call(w, codes, scales, scale=scale)
    got_c, got_s, got_out = c_d.cpu().numpy(), s_d.cpu().double().numpy(), f64(out)
    idx = w.state_indices.numpy().astype(np.int64)
    active = (idx >= 0) & (idx < w.N)
    assert (got_out[~active] == 0).all(), "inactive rows must give exactly zero"
    assert_output_close(got_out, ref_out)
    slots = idx[active]
    check_state(got_c[slots], got_s[slots], ref_c[slots], ref_s[slots], info["S_new"])
    untouched = np.setdiff1d(np.arange(w.N), slots)
    assert np.array_equal(got_c[untouched], codes.numpy()[untouched]), "untouched codes changed"
    assert np.array_equal(got_s[untouched], scales.double().numpy()[untouched]), "untouched scales changed"
    return got_c, got_s, got_out


@pytest.mark.parametrize("B", [1, 5, 32])
@pytest.mark.parametrize("config", [-1, 0, 1, 3])
def test_fp8_decode_matches_oracle(dev, B, config):
    w, codes, scales = make(B, B + 6, seed=400 + B, layout="fused" if B > 1 else "separate",
                            inactive_frac=0.2 if B > 1 else 0.0)
    run_and_check(w, codes, scales, dev, config_override=config)


def test_fp8_decode_scale_and_heads(dev):
    w, codes, scales = make(3, 5, seed=410, H=3)
    run_and_check(w, codes, scales, dev, scale=0.5, config_override=2)


def test_fp8_decode_serving_batch_sampled(dev):
    """B = 512 with ~5 % inactive rows in the fused layout: the whole call on
    the GPU, the oracle on 24 sampled rows (rows are independent)."""
    B, N = 512, 640
    w, codes, scales = make(B, N, seed=420, layout="fused", inactive_frac=0.05)
    wd = w.to(dev)
    c_d, s_d = codes.to(dev), scales.to(dev)
    out = gpu_call(wd, c_d, s_d)
    torch.cuda.synchronize()
    idx = w.state_indices.numpy().astype(np.int64)
    active = (idx >= 0) & (idx < N)
    got_out = f64(out)
    assert (got_out[~active] == 0).all()
    rows = list(np.random.default_rng(0).choice(np.nonzero(active)[0], 24, replace=False))
    ref_c, ref_s, ref_out, info = oracle_call(w, codes, scales, rows=rows)
    assert_output_close(got_out[rows], ref_out)
    slots = idx[rows]
    check_state(c_d.cpu().numpy()[slots], s_d.cpu().double().numpy()[slots], ref_c[slots], ref_s[slots],
                info["S_new"])
    untouched = np.setdiff1d(np.arange(N), idx[active])
    assert np.array_equal(c_d.cpu().numpy()[untouched], codes.numpy()[untouched])


def test_fp8_plain_path_equals_bulk_path(dev):
    """A misaligned pool (codes at a 1-byte offset, scales at a 4-byte offset)
    takes the plain-load variant: the same bits as the bulk-copy variant."""
    w, codes, scales = make(6, 9, seed=430, inactive_frac=0.2)
    wd = w.to(dev)
    c1, s1 = codes.to(dev), scales.to(dev)
    out1 = gpu_call(wd, c1, s1)
    slot, sslot = codes[0].numel(), scales[0].numel()
    cbuf = torch.zeros(codes.numel() + 16, dtype=torch.uint8, device=dev)
    sbuf = torch.zeros(scales.numel() + 4, dtype=torch.float32, device=dev)
    c2 = cbuf[1:1 + codes.numel()].view(codes.shape)
    s2 = sbuf[1:1 + scales.numel()].view(scales.shape)
    c2.copy_(codes.to(dev))
    s2.copy_(scales.to(dev))
    assert c2.data_ptr() % 16 != 0 and s2.data_ptr() % 16 != 0 and slot > 0 and sslot > 0
    out2 = gpu_call(wd, c2, s2)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(c1, c2) and torch.equal(s1, s2)


def test_fp8_graph_replay_is_deterministic(dev):
    w, codes, scales = make(32, 40, seed=440)
    wd = w.to(dev)
    c0, s0 = codes.to(dev), scales.to(dev)
    c, s = c0.clone(), s0.clone()
    out = torch.empty((32, 12, 128), dtype=torch.bfloat16, device=dev)
    gpu_call(wd, c, s, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    c.copy_(c0)
    s.copy_(s0)
    with torch.cuda.graph(g):
        gpu_call(wd, c, s, out=out)
    results = []
    for _ in range(2):
        c.copy_(c0)
        s.copy_(s0)
        g.replay()
        torch.cuda.synchronize()
        results.append((out.clone(), c.clone(), s.clone()))
    assert all(torch.equal(a, b) for a, b in zip(results[0], results[1]))


def test_fp8_chained_steps(dev):
    """Eight chained decode steps on the same slots: each side runs its own
    chain; outputs stay within the decode tolerance at every step."""
    B, N, steps = 4, 8, 8
    codes, scales = workloads.fp8_pool(N, seed=450)
    c_d, s_d = codes.to(dev), scales.to(dev)
    ref_c, ref_s = codes.numpy(), scales.double().numpy()
    for t in range(steps):
        w = workloads.decode_inputs(B, N, seed=460 + t)
        w.state_indices.copy_(torch.tensor([1, 3, 4, 6], dtype=torch.int32))
        wd = w.to(dev)
        out = gpu_call(wd, c_d, s_d)
        torch.cuda.synchronize()
        ref_c, ref_s, ref_out, _ = oracle.kda_decode_fp8(
            ref_c, ref_s, w.state_indices.numpy(), f64(w.q), f64(w.k), f64(w.v), f64(w.g_raw),
            f64(w.beta_logit), f64(w.A_log), f64(w.dt_bias), LB)
        assert_output_close(f64(out), ref_out, what=f"output of step {t}")


def test_fp8_rejects_bad_arguments(dev):
    w, codes, scales = make(2, 3, seed=470)
    wd = w.to(dev)
    c_d, s_d = codes.to(dev), scales.to(dev)
    with pytest.raises(kda.KdaError) as e:
        gpu_call(wd, c_d, s_d, config_override=4)
    assert e.value.status == kda.KDA_EUNSUPPORTED
    with pytest.raises(TypeError):
        gpu_call(wd, c_d.float(), s_d)
    out_bad = torch.empty((2, 12, 128), dtype=torch.bfloat16, device=dev)
    with pytest.raises(kda.KdaError) as e:  # out aliasing the scales
        kda.kda_decode_fp8(c_d, s_d, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit, wd.A_log,
                           wd.dt_bias, out=s_d.view(-1).view(torch.bfloat16)[:2 * 12 * 128].view(2, 12, 128))
    assert e.value.status == kda.KDA_EINVAL
    del out_bad


def test_fp8_precomputed_gate_and_empty_cases(dev):
    """The pre-computed gate convention, an empty pool (every row inactive) and
    an empty batch."""
    w = workloads.decode_inputs(4, 6, seed=480, gate_mode=1)
    codes, scales = workloads.fp8_pool(6, seed=481)
    wd = w.to(dev)
    c_d, s_d = codes.to(dev), scales.to(dev)
    out = kda.kda_decode_fp8(c_d, s_d, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit, None, None,
                             gate_mode=kda.KDA_GATE_PRECOMPUTED)
    torch.cuda.synchronize()
    ref_c, ref_s, ref_out, info = oracle.kda_decode_fp8(
        codes.numpy(), scales.double().numpy(), w.state_indices.numpy(), f64(w.q), f64(w.k), f64(w.v),
        f64(w.g_raw), f64(w.beta_logit), None, None, LB, 1.0, oracle.GATE_PRECOMPUTED)
    assert_output_close(f64(out), ref_out)
    slots = w.state_indices.numpy().astype(np.int64)
    check_state(c_d.cpu().numpy()[slots], s_d.cpu().double().numpy()[slots], ref_c[slots], ref_s[slots],
                info["S_new"])
    # N = 0: every row inactive, zero output
    empty_c, empty_s = c_d[:0], s_d[:0]
    out = torch.full((4, 12, 128), 7.0, dtype=torch.bfloat16, device=dev)
    kda.kda_decode_fp8(empty_c, empty_s, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit, None, None,
                       out=out, gate_mode=kda.KDA_GATE_PRECOMPUTED)
    torch.cuda.synchronize()
    assert not out.any()
    # B = 0: nothing happens
    before = c_d.clone()
    kda.kda_decode_fp8(c_d, s_d, wd.state_indices[:0], wd.q[:0], wd.k[:0], wd.v[:0], wd.g_raw[:0],
                       wd.beta_logit[:0], None, None, gate_mode=kda.KDA_GATE_PRECOMPUTED)
    torch.cuda.synchronize()
    assert torch.equal(before, c_d)
