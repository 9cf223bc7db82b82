"""Feeds a workloads.Problem (host copies) to the CPU oracle.

The oracle receives the generator's inputs and nothing produced by the CUDA
library: every array passed here is a fresh host copy of a generator-filled
tensor, or of an array the oracle itself wrote.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import oracle
from workloads import Problem, to_bits


@dataclass
class HostLayer:
    """Host (numpy) copies of one layer's tensors, in the oracle's types."""
    fused: np.ndarray
    A_log: np.ndarray
    dt_bias: np.ndarray
    conv_weight: np.ndarray
    conv_state: np.ndarray
    state: np.ndarray
    corr: np.ndarray
    key_gate: np.ndarray
    out: np.ndarray


def host_layer(prob: Problem, l: int, *, slots: np.ndarray | None = None) -> HostLayer:
    """Copy layer ``l`` to the host.  With ``slots`` given, only those state
    slots are copied (the rest of the host pool stays zero), which keeps the
    copy small at full size."""
    if slots is None:
        state = prob.state[l].cpu().numpy().copy()
    else:
        state = np.zeros(prob.state.shape[1:], np.float32)
        idx = np.unique(slots[slots > 0]).astype(np.int64)
        if idx.size:
            state[idx] = prob.state[l][torch.as_tensor(idx, device=prob.device)].cpu().numpy()
    return HostLayer(
        fused=to_bits(prob.fused[l]),
        A_log=prob.A_log[l].cpu().numpy(),
        dt_bias=prob.dt_bias[l].cpu().numpy(),
        conv_weight=to_bits(prob.conv_weight[l]),
        conv_state=to_bits(prob.conv_state[l]).copy(),
        state=state,
        corr=to_bits(prob.corr[l]).copy(),
        key_gate=to_bits(prob.key_gate[l]).copy(),
        out=to_bits(prob.out[l]).copy(),
    )


def run_verify(prob: Problem, hl: HostLayer, meta=None, item_mask=None, **kw):
    cfg = prob.cfg
    meta = meta or prob.meta
    H, K = cfg.H, cfg.K
    f = hl.fused
    return oracle.verify(
        H=H, K=K, Q=cfg.Q, W=cfg.W,
        mixed_qkv=f[:, : 3 * H * K], raw_gate=f[:, 3 * H * K: 4 * H * K],
        raw_beta=f[:, 4 * H * K: 4 * H * K + H],
        A_log=hl.A_log, dt_bias=hl.dt_bias, lower_bound=cfg.lower_bound,
        conv_weight=hl.conv_weight, conv_state=hl.conv_state,
        conv_dim_first=cfg.conv_dim_first, state=hl.state,
        corr=hl.corr, key_gate=hl.key_gate, out=hl.out,
        query_start_loc=meta.query_start_loc, state_indices=meta.state_indices,
        record_indices=meta.record_indices, num_accepted_prev=meta.num_accepted_prev,
        item_mask=item_mask, **kw)


def run_commit(prob: Problem, hl: HostLayer, meta=None, item_mask=None, **kw):
    cfg = prob.cfg
    meta = meta or prob.meta
    return oracle.commit(
        H=cfg.H, K=cfg.K, Q=cfg.Q, state=hl.state, corr=hl.corr, key_gate=hl.key_gate,
        A_log=hl.A_log, dt_bias=hl.dt_bias, lower_bound=cfg.lower_bound,
        query_start_loc=meta.query_start_loc, state_indices=meta.state_indices,
        num_accepted=meta.num_accepted, record_indices=meta.record_indices,
        item_mask=item_mask, **kw)
