"""The host-fed decode step with overlapped copies (workloads.drive.HostPipeline,
which bench.py's end-to-end figure runs): each layer's copies run on other
streams than its kernels, so check that a run of steps gives exactly what the
same steps give one after another with synchronous copies."""
from __future__ import annotations

import pytest
import torch

import linear_attention_ssm_kda_gb300 as kda
from linear_attention_ssm_kda_gb300 import _build
from workloads import CONFIGS, make_problem
from workloads.drive import HostPipeline, commit_all, commit_context, device_meta, pinned_meta, verify_layer

pytestmark = pytest.mark.gpu


def test_pipelined_steps_match_serial_steps():
    _build.build()
    kda.load_library()
    dev = torch.device("cuda:0")
    prob = make_problem(CONFIGS["C2"], dev, B=32, L=3, slots=64)
    L = prob.cfg.L
    ctx = commit_context(prob)
    # two different activation sets, alternated by step, so a step that read
    # the wrong (stale or early) activations would show in its outputs
    g = torch.Generator(device=dev).manual_seed(77)
    acts = [prob.fused.clone(), torch.randn(prob.fused.shape, generator=g, device=dev).to(prob.fused.dtype)]
    host_acts = [a.cpu().pin_memory() for a in acts]
    host_meta = pinned_meta(prob.meta)
    tensors = {"state": prob.state, "conv": prob.conv_state, "corr": prob.corr, "kg": prob.key_gate,
               "out": prob.out}
    start = {k: t.clone() for k, t in tensors.items()}

    steps = 5
    outs = [torch.empty(prob.out.shape, dtype=prob.out.dtype, pin_memory=True) for _ in range(steps)]
    stream = torch.cuda.current_stream(dev)
    pipe = HostPipeline(prob, ctx, stream)
    for k in range(steps):
        pipe.step(host_acts[k % 2], host_meta, outs[k])
    pipe.drain()
    torch.cuda.synchronize(dev)
    piped = {k: t.clone() for k, t in tensors.items()}

    for k, t in tensors.items():
        t.copy_(start[k])
    dm = device_meta(prob.meta, dev)
    for k in range(steps):
        prob.fused.copy_(acts[k % 2])
        for l in range(L):
            verify_layer(prob, l, dm)
        commit_all(ctx, dm)
        torch.cuda.synchronize(dev)
        assert torch.equal(prob.out.cpu().view(torch.int16), outs[k].view(torch.int16)), f"step {k} outputs"
    for k, t in tensors.items():
        a = t.view(torch.int32) if t.element_size() == 4 else t.view(torch.int16)
        b = piped[k].view(torch.int32) if t.element_size() == 4 else piped[k].view(torch.int16)
        assert torch.equal(a, b), k
    # the two activation sets did give different outputs
    assert not torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
