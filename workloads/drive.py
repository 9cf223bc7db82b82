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


def problem_scratch(prob: Problem) -> torch.Tensor:
    """The verify's device scratch for this workload, allocated once (every
    layer's verify reuses it in stream order)."""
    sc = prob.extra.get("scratch")
    if sc is None:
        cfg = prob.cfg
        sc = kda.new_verify_scratch(cfg.B, cfg.H, cfg.K, cfg.Q, prob.fused.device)
        prob.extra["scratch"] = sc
    return sc


def problem_workspace(prob: Problem) -> torch.Tensor:
    """A device workspace for this workload's verifies and commits, allocated
    once (its ticket counter is back at zero after every verify launch, so
    launches in stream order share it)."""
    ws = prob.extra.get("workspace")
    if ws is None:
        ws = kda.new_workspace(prob.fused.device)
        prob.extra["workspace"] = ws
    return ws


def verify_layer(prob: Problem, l: int, dm: DeviceMeta, *, out=None, workspace=None, stream=None,
                 fused=None, fold: DeviceMeta | None = None, variant: str = "auto", debug=None) -> None:
    """One layer's verify.  With ``fold`` (the previous step's metadata) the
    previous step's accepted records are folded into the checkpoints first,
    in the same launch (``kda_verify_fold``).  ``workspace``: the problem's
    own (``problem_workspace``) unless given."""
    cfg = prob.cfg
    H, K = cfg.H, cfg.K
    f = prob.fused[l] if fused is None else fused
    scratch = problem_scratch(prob) if f.is_cuda else None
    if workspace is None and f.is_cuda:
        workspace = problem_workspace(prob)
    kda.verify(
        mixed_qkv=f[:, : 3 * H * K], raw_gate=f[:, 3 * H * K: 4 * H * K],
        raw_beta=f[:, 4 * H * K: 4 * H * K + H],
        A_log=prob.A_log[l], dt_bias=prob.dt_bias[l], lower_bound=cfg.lower_bound,
        state=prob.state[l], correction=prob.corr[l], key_gate=prob.key_gate[l],
        query_start_loc=dm.query_start_loc, state_indices=dm.state_indices,
        num_accepted_tokens=dm.num_accepted_prev, record_indices=dm.record_indices,
        conv_state=prob.conv_state[l], conv_weight=prob.conv_weight[l],
        out=prob.out[l] if out is None else out, window=cfg.Q, conv_dim_first=cfg.conv_dim_first,
        workspace=workspace, stream=stream,
        fold_query_start_loc=None if fold is None else fold.query_start_loc,
        fold_num_accepted=None if fold is None else fold.num_accepted,
        fold_record_indices=None if fold is None else fold.record_indices,
        scratch=scratch, variant=variant, debug=debug)


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


def pinned_meta(meta: Metadata) -> dict:
    """The step's request metadata as pinned host int32 tensors."""
    return {k: torch.from_numpy(np.ascontiguousarray(v, dtype=np.int32)).pin_memory()
            for k, v in (("qsl", meta.query_start_loc), ("si", meta.state_indices),
                         ("prev", meta.num_accepted_prev), ("acc", meta.num_accepted)) if v is not None}


class HostPipeline:
    """Decode steps (verify of every layer, then the commit) fed from pinned
    host memory, with the copies of one layer overlapping the kernels of its
    neighbours.  Layer l's activations go up on one copy stream while the
    previous step's later layers run; its outputs come back on another while
    later layers run.
    Events order every reuse of a device buffer: a layer's activations are
    overwritten only after the previous step's verify of that layer, its
    outputs only after they were read back, and the request metadata
    alternates between two device sets."""

    def __init__(self, prob: Problem, ctx: kda.CommitContext, stream: torch.cuda.Stream):
        self.prob, self.ctx, self.stream = prob, ctx, stream
        dev = prob.fused.device
        L = prob.cfg.L
        self.dms = [device_meta(prob.meta, dev), device_meta(prob.meta, dev)]
        self.up = torch.cuda.Stream(dev)
        self.down = torch.cuda.Stream(dev)
        self.in_ready = [torch.cuda.Event() for _ in range(L)]
        self.verified = [torch.cuda.Event() for _ in range(L)]
        self.read_back = [torch.cuda.Event() for _ in range(L)]
        self.meta_ready = torch.cuda.Event()
        self.meta_free = [torch.cuda.Event(), torch.cuda.Event()]
        self.count = 0

    def step(self, host_fused: torch.Tensor, host_meta: dict, host_out: torch.Tensor) -> None:
        """Enqueue one step: ``host_fused`` [L, T, F] and ``host_meta`` (from
        ``pinned_meta``) in, ``host_out`` [L, T, H K] back, all pinned."""
        prob, stream, up, down = self.prob, self.stream, self.up, self.down
        L = prob.cfg.L
        d = self.dms[self.count % 2]
        with torch.cuda.stream(up):
            up.wait_event(self.meta_free[self.count % 2])  # the step two back is done with this set
            d.query_start_loc.copy_(host_meta["qsl"], non_blocking=True)
            d.state_indices.copy_(host_meta["si"], non_blocking=True)
            if "prev" in host_meta:
                d.num_accepted_prev.copy_(host_meta["prev"], non_blocking=True)
            d.num_accepted.copy_(host_meta["acc"], non_blocking=True)
            self.meta_ready.record(up)
            for l in range(L):
                up.wait_event(self.verified[l])  # the previous step's verify has read these activations
                prob.fused[l].copy_(host_fused[l], non_blocking=True)
                self.in_ready[l].record(up)
        # events of one stream complete in order: the last layer's upload of this
        # step and the last layer's read-back of the previous step cover every
        # layer, and both are done by the time the previous step's commit ends
        stream.wait_event(self.meta_ready)
        stream.wait_event(self.in_ready[L - 1])
        stream.wait_event(self.read_back[L - 1])
        for l in range(L):
            verify_layer(prob, l, d, stream=stream)
            self.verified[l].record(stream)
        commit_all(self.ctx, d, stream=stream)
        self.meta_free[self.count % 2].record(stream)
        with torch.cuda.stream(down):
            for l in range(L):
                down.wait_event(self.verified[l])
                host_out[l].copy_(prob.out[l], non_blocking=True)
                self.read_back[l].record(down)
        self.count += 1

    def drain(self) -> None:
        """Make the compute stream wait for every copy enqueued so far."""
        self.stream.wait_stream(self.up)
        self.stream.wait_stream(self.down)
