"""kda_commit_noalloc: the commit with its per-layer tables in the library's
static device scratch instead of caller-allocated device memory.

The GPU test runs it against kda_commit on two calls in a row (different
layers, tables and accepted counts), so a stale scratch would show; it must
pass alone and after the rest of the suite, so it builds its own inputs."""
from __future__ import annotations

import ctypes

import pytest
import torch

import linear_attention_ssm_kda_gb300 as kda
from linear_attention_ssm_kda_gb300 import _build
from workloads import CONFIGS, make_problem
from workloads.drive import device_meta, verify_layer

FAKE = 0x1000  # a 16-byte-aligned non-null address; never dereferenced by the rejected calls


def _args(L):
    a = kda.CommitArgs()
    a.L, a.B, a.H, a.K, a.V, a.Q = L, 3, 4, 128, 128, 4
    a.num_slots, a.num_record_rows = 8, 8
    for name in ("state_base", "state_slot_stride", "corr_base", "corr_row_stride", "kg_base",
                 "kg_row_stride", "A_log", "dt_bias", "query_start_loc", "state_indices", "num_accepted"):
        setattr(a, name, FAKE)
    return a


def test_noalloc_rejects_before_any_cuda_call():
    _build.build()
    lib = kda.load_library()
    assert lib.kda_commit_noalloc(None, None) == kda.KDA_ERR_INVALID_ARG
    a = _args(kda.NOALLOC_MAX_LAYERS + 1)
    assert lib.kda_commit_noalloc(ctypes.byref(a), None) == kda.KDA_ERR_UNSUPPORTED
    assert "static scratch of 64 layers" in kda.last_error()
    a = _args(0)
    assert lib.kda_commit_noalloc(ctypes.byref(a), None) == kda.KDA_ERR_INVALID_ARG
    a = _args(2)
    a.kg_row_stride = 0
    assert lib.kda_commit_noalloc(ctypes.byref(a), None) == kda.KDA_ERR_INVALID_ARG
    a = _args(2)
    a.B = 0
    assert lib.kda_commit_noalloc(ctypes.byref(a), None) == kda.KDA_OK


def _noalloc(prob, states, layers, num_accepted, dm):
    cfg = prob.cfg
    kda.commit_noalloc(
        states=[states[l] for l in layers], corrections=[prob.corr[l] for l in layers],
        key_gates=[prob.key_gate[l] for l in layers], A_log=prob.A_log[list(layers)].contiguous(),
        dt_bias=prob.dt_bias[list(layers)].contiguous(), lower_bound=cfg.lower_bound, window=cfg.Q,
        num_accepted_tokens=num_accepted, state_indices=dm.state_indices,
        query_start_loc=dm.query_start_loc, record_indices=dm.record_indices)


def _context(prob, states, layers):
    cfg = prob.cfg
    return kda.CommitContext([states[l] for l in layers], [prob.corr[l] for l in layers],
                             [prob.key_gate[l] for l in layers], prob.A_log[list(layers)].contiguous(),
                             prob.dt_bias[list(layers)].contiguous(), cfg.lower_bound, cfg.Q)


@pytest.mark.gpu
def test_noalloc_commit_matches_kda_commit_on_two_calls_in_a_row():
    dev = torch.device("cuda:0")
    prob = make_problem(CONFIGS["C2"], dev, B=40, L=3, slots=64)
    dm = device_meta(prob.meta, dev)
    for l in range(prob.cfg.L):
        verify_layer(prob, l, dm)
    acc1 = dm.num_accepted
    acc2 = torch.flip(dm.num_accepted, [0]).contiguous()
    calls = [((0, 1, 2), acc1), ((2, 0), acc2)]  # different layer sets, tables and counts

    ref = prob.state.clone()
    for layers, acc in calls:
        _context(prob, ref, layers).commit(acc, dm.state_indices, dm.query_start_loc,
                                           record_indices=dm.record_indices)

    got = prob.state.clone()
    # the first call on the device does the scratch set-up; a call with no
    # requests returns before it, so run one real commit on a throw-away copy
    scratch = prob.state.clone()
    _noalloc(prob, scratch, (1,), acc1, dm)
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info(dev)[0]
    allocated_before = torch.cuda.memory_allocated(dev)
    for layers, acc in calls:
        _noalloc(prob, got, layers, acc, dm)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info(dev)[0] == free_before       # no device allocation
    assert torch.cuda.memory_allocated(dev) == allocated_before  # none through torch either
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
    # and the commits did change the states they fold into
    assert not torch.equal(got.view(torch.int32), prob.state.view(torch.int32))
