"""kda_commit_align: the commit's align mode (prefix caching), final and
boundary slots, against the oracle's align-mode commit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_ssm_kda_gb300 as kda
from compare import assert_f32_close
from linear_attention_ssm_kda_gb300 import _build
from oracle_io import host_layer, run_commit
from workloads import CONFIGS, make_problem
from workloads.drive import commit_context, device_meta, verify_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("name", ["C2", "C0"])
def test_align_commit_matches_oracle(name):
    _build.build()
    kda.load_library()
    prob = make_problem(CONFIGS[name], DEV, B=40, L=2, slots=128) if name == "C2" else make_problem(
        CONFIGS[name], DEV, slots=32)
    cfg = prob.cfg
    meta = prob.meta
    B = cfg.B
    if name == "C0":  # few requests: accept every token so that each one folds
        meta.num_accepted = np.minimum(np.diff(meta.query_start_loc), cfg.Q).astype(np.int32)
    dm = device_meta(meta, DEV)
    for l in range(cfg.L):
        verify_layer(prob, l, dm)
    torch.cuda.synchronize()
    hls = [host_layer(prob, l) for l in range(cfg.L)]
    before = prob.state.cpu().numpy()

    # final slots: the source for even requests, a free slot for odd ones (one
    # of them null: nothing written); boundary slots: free or null; recovery
    # lengths before, inside and past the window
    rng = np.random.default_rng(31)
    used = {int(x) for x in meta.state_indices if x > 0}
    free = [x for x in range(1, cfg.slots) if x not in used]
    rng.shuffle(free)
    final = meta.state_indices.astype(np.int32).copy()
    bnd = np.zeros(B, np.int32)
    for b in range(B):
        if b % 2:
            final[b] = free.pop()
        if b % 3 != 2:
            bnd[b] = free.pop()
    final[1] = 0
    R = rng.choice(np.array([-1, 0, 1, 2, 3, 5], np.int32), size=B).astype(np.int32)
    dev_t = lambda a: torch.as_tensor(a, dtype=torch.int32, device=DEV)
    ws = kda.new_workspace(DEV)
    commit_context(prob).commit(dm.num_accepted, dm.state_indices, dm.query_start_loc,
                                record_indices=dm.record_indices, workspace=ws,
                                final_state_indices=dev_t(final), boundary_state_indices=dev_t(bnd),
                                boundary_recovery_lens=dev_t(R))
    assert kda.read_device_error(ws) == 0
    after = prob.state.cpu().numpy()

    lens = np.minimum(np.diff(meta.query_start_loc), cfg.Q)
    acc = np.minimum(np.maximum(meta.num_accepted, 0), lens)
    written = set()
    checked = 0
    for l in range(cfg.L):
        bex = np.full((B, cfg.H, cfg.K, cfg.K), np.nan)
        exact = run_commit(prob, hls[l], want_exact=True, final_state_indices=final, boundary_state_indices=bnd,
                           boundary_recovery_lens=R, boundary_exact=bex)
        for b in range(B):
            s = int(meta.state_indices[b])
            if s <= 0 or acc[b] == 0 or final[b] <= 0:
                continue
            written.add((l, int(final[b])))
            assert_f32_close(after[l, final[b]], exact[b], np.ones(exact[b].shape, bool),
                             what=f"{name} layer {l} request {b} final")
            if bnd[b] > 0:
                written.add((l, int(bnd[b])))
                assert_f32_close(after[l, bnd[b]], bex[b], np.ones(bex[b].shape, bool),
                                 what=f"{name} layer {l} request {b} boundary")
                if min(max(int(R[b]), 0), int(acc[b])) == 0:  # no token before the boundary
                    np.testing.assert_array_equal(after[l, bnd[b]], before[l, s])
            checked += 1
        # every slot no request wrote keeps its bits
        for x in range(cfg.slots):
            if (l, x) not in written:
                np.testing.assert_array_equal(after[l, x], before[l, x], err_msg=f"{name} layer {l} slot {x}")
    assert checked >= (20 if name == "C2" else 3)
