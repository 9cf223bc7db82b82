"""Whole decode steps captured in a CUDA graph: the library allocates nothing
and never synchronises, each verify's tensor maps travel by value in the
launch parameters, and the ticket counter that deals a verify's items (one
workspace shared by every launch of the step) is back at zero after each
launch, so a replay must write exactly what eager launches write."""
from __future__ import annotations

import pytest
import torch

import linear_attention_ssm_kda_gb300 as kda
from linear_attention_ssm_kda_gb300 import _build
from workloads import CONFIGS, make_problem
from workloads.drive import commit_all, commit_context, device_meta, verify_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _tensors(prob):
    return {"state": prob.state, "conv": prob.conv_state, "corr": prob.corr, "kg": prob.key_gate, "out": prob.out}


def _bits(t):
    return t.view(torch.int32) if t.element_size() == 4 else t.view(torch.int16)


@pytest.mark.parametrize("schedule", ["verify_then_commit", "deferred_fold"])
def test_captured_step_replays_bit_for_bit(schedule):
    _build.build()
    kda.load_library()
    prob = make_problem(CONFIGS["C2"], DEV, B=40, L=3, slots=64)
    L = prob.cfg.L
    dm = device_meta(prob.meta, DEV)
    ctx = commit_context(prob)
    ws = kda.new_workspace(DEV)

    def step():
        if schedule == "verify_then_commit":
            for l in range(L):
                verify_layer(prob, l, dm, workspace=ws)
            commit_all(ctx, dm, workspace=ws)
        else:
            for l in range(L):
                verify_layer(prob, l, dm, fold=dm, workspace=ws)

    tensors = _tensors(prob)
    start = {k: t.clone() for k, t in tensors.items()}
    step()  # eager, twice: the second step folds what the first accepted
    step()
    torch.cuda.synchronize()
    eager = {k: t.clone() for k, t in tensors.items()}

    for k, t in tensors.items():
        t.copy_(start[k])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph):
            step()
    torch.cuda.current_stream().wait_stream(side)
    # capture does not run the work: the buffers still hold the start
    torch.cuda.synchronize()
    for k, t in tensors.items():
        assert torch.equal(_bits(t), _bits(start[k])), f"capture ran {k}"
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    for k, t in tensors.items():
        assert torch.equal(_bits(t), _bits(eager[k])), f"{schedule}: replay differs in {k}"
    assert kda.read_device_error(ws) == 0
    assert ws[8:10].tolist() == [0, 0], "the ticket counter is not back at zero"
