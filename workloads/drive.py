"""Runs the CUDA library on a generated workload (tests, smoke check, bench).

Maps a ``workloads.Problem`` onto ``linear_attention_ssm_kda_gb300.verify``
and ``CommitContext.commit``; it never touches the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import linear_attention_ssm_kda_gb300 as kda
from workloads import Metadata, Problem


@dataclass
class DeviceMeta:
    query_start_loc: torch.Tensor
    state_indices: torch.Tensor
    record_indices: torch.Tensor | None
    num_accepted_prev: torch.Tensor | None
    num_accepted: torch.Tensor
    T: int


def device_meta(meta: Metadata, device) -> DeviceMeta:
    def d(a):
        return None if a is None else torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32, device=device)

    return DeviceMeta(d(meta.query_start_loc), d(meta.state_indices), d(meta.record_indices),
                      d(meta.num_accepted_prev), d(meta.num_accepted), meta.T)


def conv_state_view(prob: Problem, l: int) -> torch.Tensor:
    return prob.conv_state[l]


def verify_layer(prob: Problem, l: int, dm: DeviceMeta, *, out=None, workspace=None, stream=None,
                 fused=None) -> None:
    cfg = prob.cfg
    H, K = cfg.H, cfg.K
    f = prob.fused[l] if fused is None else fused
    kda.verify(
        mixed_qkv=f[:, : 3 * H * K], raw_gate=f[:, 3 * H * K: 4 * H * K],
        raw_beta=f[:, 4 * H * K: 4 * H * K + H],
        A_log=prob.A_log[l], dt_bias=prob.dt_bias[l], lower_bound=cfg.lower_bound,
        state=prob.state[l], correction=prob.corr[l], key_gate=prob.key_gate[l],
        query_start_loc=dm.query_start_loc, state_indices=dm.state_indices,
        num_accepted_tokens=dm.num_accepted_prev, record_indices=dm.record_indices,
        conv_state=prob.conv_state[l], conv_weight=prob.conv_weight[l],
        out=prob.out[l] if out is None else out, window=cfg.Q, conv_dim_first=cfg.conv_dim_first,
        workspace=workspace, stream=stream)


def commit_context(prob: Problem) -> kda.CommitContext:
    cfg = prob.cfg
    L = cfg.L
    return kda.CommitContext([prob.state[l] for l in range(L)], [prob.corr[l] for l in range(L)],
                             [prob.key_gate[l] for l in range(L)], prob.A_log, prob.dt_bias,
                             cfg.lower_bound, cfg.Q)


def commit_all(ctx: kda.CommitContext, dm: DeviceMeta, *, num_accepted=None, workspace=None,
               stream=None) -> None:
    ctx.commit(dm.num_accepted if num_accepted is None else num_accepted, dm.state_indices,
               dm.query_start_loc, record_indices=dm.record_indices, workspace=workspace, stream=stream)
