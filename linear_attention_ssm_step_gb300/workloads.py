"""Seeded synthetic inputs for the KDA serving step.

Shared by the tests, the bench and the smoke check; the same bytes feed the
CUDA library and the CPU oracle. This module draws random numbers and lays
them out; it holds none of the method's arithmetic.

Distributions (the serving workloads these stand in for; no dataset exists):
  state ~ N(0, 0.02^2) bf16; q, k, v, g_raw, beta_logit ~ N(0, 1) bf16 (pre-computed
  gate convention: g = -5 U[0, 1) and beta = U[0, 1), bf16);
  A_log = log U[1, 16] fp32 [H]; dt_bias ~ N(0, 0.5^2) fp32 [H, 128];
  ring: k_cache = unit vectors (normalised Gaussians) in bf16,
  u_cache ~ N(0, 0.5^2) bf16, g_cache = fp32 running sums over ring
  positions of increments drawn from U[-5, 0], hist_len per slot.
  prefill: packed sequences of given lengths, one token per activation row
  (the decode distributions), cu_seqlens their running offsets, one distinct
  slot per sequence (a fraction of them inactive, as for decode rows).
  fp8 state pool: E4M3 codes drawn field by field - sign uniform, exponent
  field round(N(11, 2^2)) clipped to 1..15, mantissa uniform (at most 6 when
  the exponent field is 15, so never NaN) - and per-row scales 2^e with e
  uniform in -14..-8 (row values up to 448 * 2^-8 = 1.75, typically ~0.01).
Standard deviations are given as the second argument of N(mean, sd^2).
"""

from dataclasses import dataclass, field, replace

import numpy as np
import torch

H_DEFAULT = 12
D = 128  # K = V = 128


def _gen(seed):
    return torch.Generator().manual_seed(int(seed))


def _randn(g, shape, std=1.0, dtype=torch.bfloat16):
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(dtype)


@dataclass
class Workload:
    """Inputs of one call. q, k, v are views into `qkv` when a fused layout is used."""

    state: torch.Tensor          # bf16 [N, H, 128, 128]
    state_indices: torch.Tensor  # int32 [B]
    g_raw: torch.Tensor          # bf16 [B, (T,) H, 128]
    beta_logit: torch.Tensor     # bf16 [B, (T,) H]
    A_log: torch.Tensor          # fp32 [H]
    dt_bias: torch.Tensor        # fp32 [H, 128]
    T: object = None             # None for decode, else the token count
    layout: str = "separate"     # "separate", "packed" or "fused"
    qkv: torch.Tensor = None     # packed / fused buffer [B, (T,) row]
    q_sep: torch.Tensor = None
    k_sep: torch.Tensor = None
    v_sep: torch.Tensor = None
    ring: dict = field(default_factory=dict)  # k_cache, u_cache, g_cache, hist_len, W, flush_min
    gate_mode: int = 0           # 0: raw gate and beta logits; 1: log-space g and beta given
    cu_seqlens: torch.Tensor = None  # prefill: int32 [S + 1] row offsets of the sequences

    @property
    def B(self):
        return self.state_indices.shape[0]

    @property
    def H(self):
        return self.state.shape[1]

    @property
    def N(self):
        return self.state.shape[0]

    def _part(self, i):
        if self.layout == "separate":
            return (self.q_sep, self.k_sep, self.v_sep)[i]
        hk = self.H * D
        return self.qkv[..., i * hk:(i + 1) * hk].unflatten(-1, (self.H, D))

    @property
    def q(self):
        return self._part(0)

    @property
    def k(self):
        return self._part(1)

    @property
    def v(self):
        return self._part(2)

    def select_rows(self, rows):
        """The same call restricted to batch rows `rows` (same pool and ring)."""
        rows = torch.as_tensor(rows, dtype=torch.long)
        pick = lambda t: None if t is None else t[rows]  # noqa: E731
        return replace(self, state_indices=self.state_indices[rows], g_raw=self.g_raw[rows],
                       beta_logit=self.beta_logit[rows], qkv=pick(self.qkv), q_sep=pick(self.q_sep),
                       k_sep=pick(self.k_sep), v_sep=pick(self.v_sep))

    def to(self, device):
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        ring = {k: (mv(v) if isinstance(v, torch.Tensor) else v) for k, v in self.ring.items()}
        return replace(self, state=mv(self.state), state_indices=mv(self.state_indices),
                       g_raw=mv(self.g_raw), beta_logit=mv(self.beta_logit), A_log=mv(self.A_log),
                       dt_bias=mv(self.dt_bias), qkv=mv(self.qkv), q_sep=mv(self.q_sep),
                       k_sep=mv(self.k_sep), v_sep=mv(self.v_sep), ring=ring, cu_seqlens=mv(self.cu_seqlens))

    def clone(self):
        c = lambda t: None if t is None else t.clone()  # noqa: E731
        ring = {k: (c(v) if isinstance(v, torch.Tensor) else v) for k, v in self.ring.items()}
        return replace(self, state=c(self.state), state_indices=c(self.state_indices),
                       g_raw=c(self.g_raw), beta_logit=c(self.beta_logit), A_log=c(self.A_log),
                       dt_bias=c(self.dt_bias), qkv=c(self.qkv), q_sep=c(self.q_sep),
                       k_sep=c(self.k_sep), v_sep=c(self.v_sep), ring=ring, cu_seqlens=c(self.cu_seqlens))


def slot_indices(g, B, N, inactive_frac=0.0):
    """B distinct slots of a pool of N; a fraction of rows made inactive
    (half negative, half >= N)."""
    n_inactive = int(round(inactive_frac * B))
    n_active = B - n_inactive
    if n_active > N:
        raise ValueError(f"{n_active} active rows need a pool of at least that many slots, got {N}")
    idx = torch.randperm(N, generator=g)[:n_active].to(torch.int64)
    bad = []
    for i in range(n_inactive):
        r = int(torch.randint(0, 1000, (1,), generator=g))
        bad.append(-1 - r if i % 2 == 0 else N + r)
    idx = torch.cat([idx, torch.tensor(bad, dtype=torch.int64)])
    perm = torch.randperm(B, generator=g)
    return idx[perm].to(torch.int32)


def decode_inputs(B, N, seed=0, T=None, layout="separate", inactive_frac=0.0, H=H_DEFAULT,
                  state_std=0.02, indices=None, gate_mode=0):
    """Inputs of kda_decode (T None) or kda_verify (T tokens).

    layout "packed": one bf16 row [3][H][128] per (b, t), as a serving stack's
    QKV projection writes it; "fused": the same row followed by 64 more
    columns ([B, 3*H*128 + 64]), so q, k, v are strided views of a wider
    projection buffer; "separate": three contiguous tensors.
    """
    g = _gen(seed)
    tok = () if T is None else (T,)
    state = _randn(g, (N, H, D, D), state_std)
    if indices is None:
        indices = slot_indices(g, B, N, inactive_frac)
    hk = H * D
    kw = {}
    if layout == "separate":
        kw.update(q_sep=_randn(g, (B,) + tok + (H, D)), k_sep=_randn(g, (B,) + tok + (H, D)),
                  v_sep=_randn(g, (B,) + tok + (H, D)))
    elif layout == "packed":
        kw.update(qkv=_randn(g, (B,) + tok + (3 * hk,)))
    elif layout == "fused":
        kw.update(qkv=_randn(g, (B,) + tok + (3 * hk + 64,)))
    else:
        raise ValueError(layout)
    if gate_mode == 1:  # pre-computed convention: log-space g in [-5, 0), beta in [0, 1)
        g_in = (-5.0 * torch.rand((B,) + tok + (H, D), generator=g)).to(torch.bfloat16)
        b_in = torch.rand((B,) + tok + (H,), generator=g).to(torch.bfloat16)
    else:
        g_in, b_in = _randn(g, (B,) + tok + (H, D)), _randn(g, (B,) + tok + (H,))
    return Workload(
        state=state, state_indices=torch.as_tensor(indices, dtype=torch.int32),
        g_raw=g_in, beta_logit=b_in, gate_mode=gate_mode,
        A_log=torch.log(torch.rand((H,), generator=g, dtype=torch.float32) * 15.0 + 1.0),
        dt_bias=torch.randn((H, D), generator=g, dtype=torch.float32) * 0.5,
        T=T, layout=layout, **kw)


def ring_inputs(B, N, T, W=32, flush_min=9, fold_frac=0.0, seed=0, H=H_DEFAULT, layout="separate",
                inactive_frac=0.0, sentinels=True, gate_mode=0, circular=False):
    """Inputs of kda_verify_ring. Active rows fold with probability given by
    fold_frac (exactly round(fold_frac * active) of them): their hist_len is
    drawn from [flush_min, flush_min + T - 1], the others' from [0, flush_min - 1].
    Ring positions at or past hist_len hold NaN, so a stray read shows up.
    circular: every slot gets a random ring start cache_base in [0, W), and its
    ring is stored rotated by it (position P at entry (cache_base + P) mod W)."""
    w = decode_inputs(B, N, seed=seed, T=T, layout=layout, inactive_frac=inactive_frac, H=H, gate_mode=gate_mode)
    g = _gen(seed + 7919)
    x = torch.randn((N, H, W, D), generator=g, dtype=torch.float64)
    k_cache = (x / x.norm(dim=-1, keepdim=True)).to(torch.bfloat16)
    u_cache = _randn(g, (N, H, W, D), 0.5)
    inc = -5.0 * torch.rand((N, H, W, D), generator=g, dtype=torch.float32)
    g_cache = torch.from_numpy(np.cumsum(inc.numpy(), axis=2, dtype=np.float32))
    hist = torch.randint(0, flush_min, (N,), generator=g, dtype=torch.int32)
    idx = w.state_indices.to(torch.int64)
    active = [int(n) for n in idx if 0 <= n < N]
    n_fold = int(round(fold_frac * len(active)))
    perm = torch.randperm(len(active), generator=g)
    for i, j in enumerate(perm.tolist()):
        n = active[j]
        if i < n_fold:
            hist[n] = int(torch.randint(flush_min, flush_min + T, (1,), generator=g))
        else:
            hist[n] = int(torch.randint(0, flush_min, (1,), generator=g))
    if sentinels:
        pos = torch.arange(W).view(1, 1, W, 1)
        dead = pos >= hist.view(N, 1, 1, 1).to(torch.int64)
        k_cache = k_cache.masked_fill(dead, float("nan"))
        u_cache = u_cache.masked_fill(dead, float("nan"))
        g_cache = g_cache.masked_fill(dead, float("nan"))
    cache_base = None
    if circular:
        cache_base = torch.randint(0, W, (N,), generator=g, dtype=torch.int32)
        shifts = [int(c) for c in cache_base]
        k_cache = torch.stack([torch.roll(k_cache[n], shifts[n], dims=1) for n in range(N)])
        u_cache = torch.stack([torch.roll(u_cache[n], shifts[n], dims=1) for n in range(N)])
        g_cache = torch.stack([torch.roll(g_cache[n], shifts[n], dims=1) for n in range(N)])
    w.ring = dict(k_cache=k_cache, u_cache=u_cache, g_cache=g_cache, hist_len=hist, W=W,
                  flush_min=flush_min, cache_base=cache_base)
    return w


def prefill_inputs(lengths, N, seed=0, layout="separate", inactive_frac=0.0, H=H_DEFAULT, state_std=0.02,
                   gate_mode=0):
    """Inputs of kda_prefill: len(lengths) sequences packed row after row
    (L = sum(lengths) activation rows, drawn as decode rows), cu_seqlens their
    offsets, state_indices one slot per sequence (some inactive)."""
    L = int(sum(lengths))
    g = _gen(seed + 104729)
    idx = slot_indices(g, len(lengths), N, inactive_frac)
    w = decode_inputs(L, N, seed=seed, layout=layout, H=H, state_std=state_std, gate_mode=gate_mode,
                      indices=torch.zeros(L, dtype=torch.int32))
    w.state_indices = idx
    w.cu_seqlens = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    return w


def fp8_pool(N, H=H_DEFAULT, seed=0):
    """An fp8 (E4M3) state pool: codes uint8 [N, H, 128, 128] and fp32 row
    scales [N, H, 128] (powers of two), drawn as in the module docstring."""
    g = _gen(seed)
    shape = (N, H, D, D)
    sign = torch.randint(0, 2, shape, generator=g, dtype=torch.int64)
    ef = torch.clamp(torch.round(torch.randn(shape, generator=g) * 2.0 + 11.0), 1, 15).to(torch.int64)
    mant = torch.randint(0, 8, shape, generator=g, dtype=torch.int64)
    mant = torch.where(ef == 15, torch.clamp(mant, max=6), mant)
    codes = ((sign << 7) | (ef << 3) | mant).to(torch.uint8)
    e = torch.randint(-14, -7, (N, H, D), generator=g, dtype=torch.int64)
    scales = torch.pow(2.0, e.to(torch.float64)).to(torch.float32)
    return codes, scales
