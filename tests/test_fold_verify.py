"""kda_verify_fold: the previous step's accepted records folded into each
checkpoint inside the verify (the deferred form of the hot path, one launch
per layer instead of a commit launch plus a verify launch).  The oracle runs
the definition: the commit of the previous step, then the verify."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_ssm_kda_gb300 as kda
from compare import assert_bf16_outputs, assert_f32_close, assert_same_written, written_bf16
from linear_attention_ssm_kda_gb300 import _build
from oracle_io import host_layer, run_commit, run_verify
from test_parity_gpu import check_commit_layer
from workloads import CONFIGS, Metadata, canary_fill_, make_problem, next_step_metadata, to_bits
from workloads.drive import device_meta, verify_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    kda.load_library()


def _drop_windows(meta: Metadata, rows: np.ndarray) -> Metadata:
    """The same step with the windows of ``rows`` emptied (nothing to verify,
    nothing accepted): their pending records are then folded only."""
    lens = np.diff(meta.query_start_loc).astype(np.int64)
    lens[rows] = 0
    qsl = np.zeros(lens.size + 1, np.int32)
    qsl[1:] = np.cumsum(lens)
    acc = meta.num_accepted.copy()
    acc[rows] = 0
    return Metadata(qsl, meta.state_indices.copy(),
                    None if meta.record_indices is None else meta.record_indices.copy(),
                    meta.num_accepted_prev.copy(), acc)


def _check_step(prob, l, hl, res, what):
    """Outputs (written set and values), key/gate records and conv state bit
    for bit, and this step's corrections against the oracle's exact values.
    The records are not canary-filled: the fold reads the pending ones."""
    g_out = to_bits(prob.out[l])
    out_m = written_bf16(hl.out)
    assert_same_written(written_bf16(g_out), out_m, f"{what} out")
    assert_bf16_outputs(g_out, hl.out, res["out_exact"], out_m, what=f"{what} out")
    np.testing.assert_array_equal(to_bits(prob.key_gate[l]), hl.key_gate, err_msg=f"{what} key_gate bits")
    np.testing.assert_array_equal(to_bits(prob.conv_state[l]), hl.conv_state, err_msg=f"{what} conv state bits")
    corr_m = ~np.isnan(res["corr_exact"])
    assert_f32_close(prob.corr[l].cpu().numpy(), res["corr_exact"], corr_m, what=f"{what} corr")


@pytest.mark.parametrize("name", ["C4", "C0", "C3", "C0-Q6"])
def test_fold_chain_matches_commit_then_verify(name):
    """Three decode steps.  Step 0 is a plain verify; steps 1 and 2 fold the
    previous step's accepted tokens and verify in one launch per layer.  Step
    2 empties three windows, so those requests are folded only.  C4 brings
    null slots and activation rows at 8-byte offsets; C0 the K = 64 build;
    C3 windows of 8 tokens with the lower-bound gate and outliers; C0-Q6 a
    window of 6 on the window-of-8 build."""
    if name == "C4":
        prob = make_problem(CONFIGS[name], DEV, B=96, L=2, slots=256)
    elif name == "C3":
        prob = make_problem(CONFIGS[name], DEV, B=48, L=2, slots=128)
    elif name == "C0-Q6":
        prob = make_problem(CONFIGS["C0"].replace(Q=6), DEV)
    else:
        prob = make_problem(CONFIGS[name], DEV)
    cfg = prob.cfg
    rng = np.random.default_rng(2024)
    hls = [host_layer(prob, l) for l in range(cfg.L)]
    ws = kda.new_workspace(DEV)
    meta_prev = None
    folded_only = 0
    for step in range(3):
        meta = prob.meta if step == 0 else next_step_metadata(prob, rng)
        if step == 2:
            n_prev = np.minimum(np.diff(meta_prev.query_start_loc), cfg.Q)
            pending = np.minimum(np.maximum(meta_prev.num_accepted, 0), n_prev)
            rows = np.flatnonzero((meta.state_indices > 0) & (pending > 0))[:3]
            folded_only = rows.size
            meta = _drop_windows(meta, rows)
        if step > 0:
            g = torch.Generator(device=DEV).manual_seed(500 + step)
            prob.fused = torch.randn((cfg.L, meta.T, prob.fused.shape[2]), generator=g, device=DEV).to(torch.bfloat16)
            prob.out = torch.empty((cfg.L, meta.T, cfg.H * cfg.K), dtype=torch.bfloat16, device=DEV)
            for l in range(cfg.L):
                hls[l].fused = to_bits(prob.fused[l])
                hls[l].out = np.empty((meta.T, cfg.H * cfg.K), np.uint16)
        prob.meta = meta
        canary_fill_(prob.out)
        for l in range(cfg.L):
            hls[l].out[...] = 0x7FA5
        gpu_before = prob.state.cpu().numpy()
        dm = device_meta(meta, DEV)
        dmp = None if meta_prev is None else device_meta(meta_prev, DEV)
        for l in range(cfg.L):
            verify_layer(prob, l, dm, workspace=ws, fold=dmp)
        assert kda.read_device_error(ws) == 0
        for l in range(cfg.L):
            if meta_prev is not None:
                exact = run_commit(prob, hls[l], meta=meta_prev, want_exact=True)
                check_commit_layer(prob, l, hls[l], exact, meta_prev, before=gpu_before[l])
            else:  # a plain verify leaves the checkpoint as it was
                np.testing.assert_array_equal(prob.state[l].cpu().numpy(), gpu_before[l])
            res = run_verify(prob, hls[l], meta=meta, want_exact=True)
            _check_step(prob, l, hls[l], res, f"{name} step {step} layer {l}")
        meta_prev = meta
    assert folded_only > 0


def test_fold_only_step_with_no_token_rows():
    """Every window of the step empty (T = 0): the pending records are folded
    and nothing else is written."""
    prob = make_problem(CONFIGS["C0"], DEV)
    cfg = prob.cfg
    meta0 = prob.meta
    meta0.num_accepted = np.minimum(np.diff(meta0.query_start_loc), cfg.Q).astype(np.int32)  # all accepted
    dm0 = device_meta(meta0, DEV)
    verify_layer(prob, 0, dm0)
    hl = host_layer(prob, 0)
    gpu_before = prob.state.cpu().numpy()
    conv_before = prob.conv_state.clone()
    B = cfg.B
    empty = Metadata(np.zeros(B + 1, np.int32), meta0.state_indices.copy(), meta0.record_indices,
                     meta0.num_accepted.copy(), np.zeros(B, np.int32))
    prob.meta = empty
    prob.fused = torch.empty((cfg.L, 0, prob.fused.shape[2]), dtype=torch.bfloat16, device=DEV)
    prob.out = torch.empty((cfg.L, 0, cfg.H * cfg.K), dtype=torch.bfloat16, device=DEV)
    ws = kda.new_workspace(DEV)
    verify_layer(prob, 0, device_meta(empty, DEV), workspace=ws, fold=dm0)
    assert kda.read_device_error(ws) == 0
    exact = run_commit(prob, hl, meta=meta0, want_exact=True)
    assert check_commit_layer(prob, 0, hl, exact, meta0, before=gpu_before[0]) is not None
    assert torch.equal(prob.conv_state.view(torch.int16), conv_before.view(torch.int16))
