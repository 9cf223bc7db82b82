"""Seeded synthetic inputs for the KDA RecoverSSM verify / commit workloads.

This module only draws random numbers and lays them out in device or host
memory.  It holds none of the method's arithmetic, so both the CUDA path and
the CPU oracle can take their inputs from it.

Draw recipe (fixed order; N(mu, sd) takes the standard deviation; a bf16
input is the round-to-nearest-even of an fp32 draw):
  * integer metadata comes from ``numpy.random.default_rng(seed)``:
    query lengths, live slots, null positions, record rows, conv offsets
    (``num_accepted_prev``) and accepted counts, in that order;
  * floating-point tensors come from a ``torch.Generator`` seeded with the same
    seed on the target device, in this order: fused projection rows
    (mixed_qkv | raw_gate | raw_beta | pad), A_log, dt_bias, conv weight,
    conv state, SSM state.

The five named workloads follow the benchmark descriptions (tiny, decode
verify, verify-then-commit over 24 layers, long window with the bounded gate
and outliers, deferred-commit stress with misaligned rows and null slots).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Config:
    name: str
    B: int                 # requests
    H: int                 # heads
    K: int                 # head dim (K == V)
    Q: int                 # speculative window (spec_query_len)
    L: int                 # KDA layers
    slots: int             # state-pool slots per layer
    seed: int
    W: int = 4             # conv width
    lower_bound: float | None = None   # None: softplus gate
    conv_dim_first: bool = True
    conv_weight_fp32: bool = False
    act_std: float = 1.0
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    state_std: float = 0.1
    null_frac: float = 0.0
    null_count: int = 0    # exact number of null requests (overrides null_frac)
    odd_start_frac: float = 0.0     # share of requests starting on an odd token row
    record_by_request: bool = False  # records indexed by a request row, not the slot
    conv_offsets: bool = True        # pass num_accepted_prev (conv read offset)
    steps: int = 1                   # deferred-commit steps (C4)

    @property
    def V(self) -> int:
        return self.K

    @property
    def conv_len(self) -> int:
        return self.Q + self.W - 2

    @property
    def conv_dim(self) -> int:
        return 3 * self.H * self.K

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


CONFIGS: dict[str, Config] = {
    # Tiny verify+commit, seed 0.
    "C0": Config("C0", B=4, H=4, K=64, Q=4, L=1, slots=8, seed=0, state_std=0.1),
    # Decode verify: 64 requests, 32 heads, seq-first conv state, 4 null slots.
    "C1": Config("C1", B=64, H=32, K=128, Q=4, L=1, slots=256, seed=1, state_std=0.05,
                 conv_dim_first=False, null_count=4),
    # Verify then commit over 24 layers.
    "C2": Config("C2", B=256, H=32, K=128, Q=4, L=24, slots=512, seed=2, state_std=0.1),
    # Long window, bounded gate, heavy-tailed activations.
    "C3": Config("C3", B=512, H=32, K=128, Q=8, L=1, slots=1024, seed=3, lower_bound=-5.0,
                 act_std=2.0, outlier_frac=0.01, outlier_scale=10.0, state_std=0.1),
    # Deferred commit stress: odd (8-byte aligned) token rows, null slots.
    "C4": Config("C4", B=1024, H=16, K=128, Q=4, L=12, slots=2048, seed=4, null_frac=0.05,
                 odd_start_frac=0.25, record_by_request=True, steps=3),
}


@dataclass
class Metadata:
    """Per-step request metadata (host numpy int32)."""
    query_start_loc: np.ndarray
    state_indices: np.ndarray
    record_indices: np.ndarray | None
    num_accepted_prev: np.ndarray | None
    num_accepted: np.ndarray

    @property
    def T(self) -> int:
        return int(self.query_start_loc[-1])


@dataclass
class Problem:
    cfg: Config
    device: torch.device
    meta: Metadata
    fused: torch.Tensor            # [L, T, F] bf16 projection rows
    A_log: torch.Tensor            # [L, H] fp32
    dt_bias: torch.Tensor          # [L, H*K] fp32
    conv_weight: torch.Tensor      # [L, 3HK, W] bf16 or fp32
    conv_state: torch.Tensor       # [L, slots, 3HK, Lc] or [L, slots, Lc, 3HK] bf16
    state: torch.Tensor            # [L, slots, H, V, K] fp32
    corr: torch.Tensor             # [L, rows, H, Q, V] fp32
    key_gate: torch.Tensor         # [L, rows, H, Q, 2K] bf16
    out: torch.Tensor              # [L, T, HV] bf16
    extra: dict = field(default_factory=dict)

    # column windows of the fused projection buffer
    def mixed_qkv(self, l: int) -> torch.Tensor:
        c = self.cfg
        return self.fused[l, :, : 3 * c.H * c.K]

    def raw_gate(self, l: int) -> torch.Tensor:
        c = self.cfg
        return self.fused[l, :, 3 * c.H * c.K: 4 * c.H * c.K]

    def raw_beta(self, l: int) -> torch.Tensor:
        c = self.cfg
        return self.fused[l, :, 4 * c.H * c.K: 4 * c.H * c.K + c.H]

    @property
    def num_record_rows(self) -> int:
        return int(self.corr.shape[1])


def fused_width(cfg: Config) -> int:
    """Row length (elements) of the fused projection buffer.  Rows are padded
    to a 16-byte multiple, except when odd rows must be 8-byte aligned only:
    then the row is 8 bytes past a 16-byte multiple."""
    F = 4 * cfg.H * cfg.K + cfg.H
    if cfg.odd_start_frac > 0:
        F += (4 - F % 8) % 8  # F % 8 == 4 -> 2F % 16 == 8
    else:
        F += (8 - F % 8) % 8
    return F


def draw_metadata(cfg: Config, rng: np.random.Generator, B: int | None = None) -> Metadata:
    B = cfg.B if B is None else B
    Q = cfg.Q
    # query lengths
    if cfg.odd_start_frac > 0:
        want_odd = rng.random(B) < cfg.odd_start_frac
        lens = np.empty(B, np.int64)
        pos = 0
        for b in range(B - 1):
            parity = (int(want_odd[b + 1]) - pos) % 2
            choices = [x for x in range(1, Q + 1) if x % 2 == parity]
            lens[b] = choices[int(rng.integers(len(choices)))]
            pos += int(lens[b])
        lens[B - 1] = int(rng.integers(1, Q + 1))
    else:
        lens = rng.integers(1, Q + 1, size=B)
    qsl = np.zeros(B + 1, np.int32)
    qsl[1:] = np.cumsum(lens)
    # live slots (slot 0 is the null block and never live)
    slots = rng.choice(np.arange(1, cfg.slots), size=B, replace=False).astype(np.int32)
    n_null = cfg.null_count if cfg.null_count else int(round(cfg.null_frac * B))
    if n_null:
        pos = rng.choice(B, size=n_null, replace=False)
        for i, p in enumerate(pos):
            slots[p] = 0 if i % 2 == 0 else -1
    rec = None
    if cfg.record_by_request:
        rec = rng.permutation(B).astype(np.int32)
    prev = rng.integers(1, Q + 1, size=B).astype(np.int32) if cfg.conv_offsets else None
    acc = np.array([rng.integers(0, l + 1) for l in np.minimum(lens, Q)], np.int32)
    return Metadata(qsl, slots, rec, prev, acc)


def _normal_bf16(gen, shape, std, device, outlier_frac=0.0, outlier_scale=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std
    if outlier_frac > 0:
        mask = torch.rand(shape, generator=gen, device=device) < outlier_frac
        x = torch.where(mask, x * outlier_scale, x)
    return x.to(torch.bfloat16)


def make_problem(cfg: Config, device="cpu", *, B: int | None = None, L: int | None = None,
                 slots: int | None = None, seed: int | None = None) -> Problem:
    """Allocate and fill every tensor of one workload on ``device``.

    ``B``, ``L`` and ``slots`` shrink the workload for tests the oracle must
    finish in seconds; every other property (distributions, layouts,
    alignment pattern) stays the configuration's."""
    if B is not None or L is not None or slots is not None:
        cfg = cfg.replace(B=B or cfg.B, L=L or cfg.L, slots=slots or cfg.slots,
                          null_count=min(cfg.null_count, B or cfg.B))
    seed = cfg.seed if seed is None else seed
    device = torch.device(device)
    rng = np.random.default_rng(seed)
    meta = draw_metadata(cfg, rng)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    H, K, Q, W, Lyr = cfg.H, cfg.K, cfg.Q, cfg.W, cfg.L
    T = meta.T
    F = fused_width(cfg)
    fused = _normal_bf16(gen, (Lyr, T, F), cfg.act_std, device, cfg.outlier_frac, cfg.outlier_scale)
    # raw_gate and raw_beta are N(0,1) regardless of the activation spread
    gb = _normal_bf16(gen, (Lyr, T, H * K + H), 1.0, device)
    fused[:, :, 3 * H * K: 4 * H * K + H] = gb
    A_log = (torch.rand((Lyr, H), generator=gen, device=device) * 2.0 - 1.0).float()
    dt_bias = (torch.randn((Lyr, H * K), generator=gen, device=device) * 0.1).float()
    cw = torch.randn((Lyr, 3 * H * K, W), generator=gen, device=device) * 0.5
    conv_weight = cw.float() if cfg.conv_weight_fp32 else cw.to(torch.bfloat16)
    cshape = ((Lyr, cfg.slots, 3 * H * K, cfg.conv_len) if cfg.conv_dim_first
              else (Lyr, cfg.slots, cfg.conv_len, 3 * H * K))
    conv_state = _normal_bf16(gen, cshape, 1.0, device)
    state = torch.randn((Lyr, cfg.slots, H, K, K), generator=gen, device=device,
                        dtype=torch.float32) * cfg.state_std
    rows = cfg.B if cfg.record_by_request else cfg.slots
    corr = torch.zeros((Lyr, rows, H, Q, K), device=device, dtype=torch.float32)
    key_gate = torch.zeros((Lyr, rows, H, Q, 2 * K), device=device, dtype=torch.bfloat16)
    out = torch.zeros((Lyr, T, H * K), device=device, dtype=torch.bfloat16)
    return Problem(cfg, device, meta, fused, A_log, dt_bias, conv_weight, conv_state,
                   state, corr, key_gate, out)


def next_step_metadata(prob: Problem, rng: np.random.Generator) -> Metadata:
    """A following decode step for the same requests: new query lengths and
    accepted counts; the conv offset of the new step is the previous step's
    accepted count (at least one token is always accepted)."""
    cfg = prob.cfg
    old = prob.meta
    B = old.state_indices.shape[0]
    lens = rng.integers(1, cfg.Q + 1, size=B)
    if cfg.odd_start_frac > 0:
        fresh = draw_metadata(cfg.replace(null_count=0, null_frac=0.0), rng, B=B)
        qsl = fresh.query_start_loc
        lens = np.diff(qsl)
    else:
        qsl = np.zeros(B + 1, np.int32)
        qsl[1:] = np.cumsum(lens)
    prev = old.num_accepted.astype(np.int32).copy()
    acc = np.array([rng.integers(0, l + 1) for l in np.minimum(lens, cfg.Q)], np.int32)
    return Metadata(qsl.astype(np.int32), old.state_indices.copy(),
                    None if old.record_indices is None else old.record_indices.copy(),
                    prev, acc)


def canary_fill_(t: torch.Tensor) -> torch.Tensor:
    """Fill a buffer with a NaN bit pattern so untouched elements are visible."""
    if t.dtype == torch.bfloat16:
        t.view(torch.int16).fill_(0x7FA5)
    elif t.dtype == torch.float32:
        t.view(torch.int32).fill_(0x7FC0DEAD)
    else:
        raise TypeError(t.dtype)
    return t


def to_bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of a tensor: bf16 as uint16 bit patterns."""
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()
