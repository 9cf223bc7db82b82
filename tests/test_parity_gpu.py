"""Parity of the CUDA library (through the C ABI) with the CPU oracle on the
five workloads, element by element at sizes the oracle finishes in seconds,
and on sampled work items at the full benchmark sizes.  Comparison rules:
tests/compare.py."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_ssm_kda_gb300 as kda
from compare import (assert_bf16_outputs, assert_f32_close, assert_same_written, written_bf16,
                     written_f32)
from linear_attention_ssm_kda_gb300 import _build
from oracle_io import host_layer, run_commit, run_verify
from workloads import CONFIGS, Config, canary_fill_, make_problem, next_step_metadata, to_bits
from workloads.drive import commit_all, commit_context, device_meta, verify_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    kda.load_library()


# --------------------------------------------------------------------------- helpers

def _item_mask(prob, n_items, seed):
    B, H = prob.cfg.B, prob.cfg.H
    rng = np.random.default_rng(seed)
    mask = np.zeros(B * H, np.uint8)
    mask[rng.choice(B * H, size=min(n_items, B * H), replace=False)] = 1
    return mask


def _masks_for_items(prob, meta, mask):
    """Element masks (out rows, record rows, conv channels) of the selected items."""
    cfg = prob.cfg
    H, K, Q = cfg.H, cfg.K, cfg.Q
    T = meta.T
    out_m = np.zeros((T, H * K), bool)
    rows = prob.num_record_rows
    rec_m = np.zeros((rows, H), bool)
    conv_m = np.zeros((cfg.slots, 3 * H * K), bool)
    for it in np.flatnonzero(mask):
        b, h = divmod(int(it), H)
        bos = int(meta.query_start_loc[b])
        n = min(int(meta.query_start_loc[b + 1]) - bos, Q)
        if n <= 0:
            continue
        out_m[bos: bos + n, h * K:(h + 1) * K] = True
        s = int(meta.state_indices[b])
        if s <= 0:
            continue
        r = s if meta.record_indices is None else int(meta.record_indices[b])
        rec_m[r, h] = True
        for g in range(3):
            conv_m[s, g * H * K + h * K: g * H * K + (h + 1) * K] = True
    return out_m, rec_m, conv_m


def _conv_as_channels(cs, dim_first):
    """[slots, C, Lc] view of either conv layout."""
    return cs if dim_first else np.swapaxes(cs, 1, 2)


def check_verify_layer(prob, l, hl, res, meta, mask=None, stats=None):
    """Compare the GPU's layer-l verify outputs with the oracle's (hl / res)."""
    cfg = prob.cfg
    g_out = to_bits(prob.out[l])
    g_corr = prob.corr[l].cpu().numpy()
    g_kg = to_bits(prob.key_gate[l])
    g_cs = to_bits(prob.conv_state[l])
    if mask is None:
        out_m = written_bf16(hl.out)
        assert_same_written(written_bf16(g_out), out_m, f"layer {l} out")
        assert_same_written(written_f32(g_corr), written_f32(hl.corr), f"layer {l} corr")
        assert_same_written(written_bf16(g_kg), written_bf16(hl.key_gate), f"layer {l} key_gate")
        corr_m = written_f32(hl.corr)
        np.testing.assert_array_equal(g_kg, hl.key_gate, err_msg=f"layer {l} key_gate bits")
        np.testing.assert_array_equal(g_cs, hl.conv_state, err_msg=f"layer {l} conv state bits")
    else:
        out_m, rec_m, conv_m = _masks_for_items(prob, meta, mask)
        corr_m = written_f32(hl.corr) & rec_m[:, :, None, None]
        kg_m = written_bf16(hl.key_gate) & rec_m[:, :, None, None]
        assert written_bf16(g_out)[out_m].all() and written_bf16(hl.out)[out_m].all()
        assert written_f32(g_corr)[corr_m].all()
        np.testing.assert_array_equal(g_kg[kg_m], hl.key_gate[kg_m], err_msg=f"layer {l} key_gate bits")
        gc = _conv_as_channels(g_cs, cfg.conv_dim_first)
        oc = _conv_as_channels(hl.conv_state, cfg.conv_dim_first)
        np.testing.assert_array_equal(gc[conv_m], oc[conv_m], err_msg=f"layer {l} conv state bits")
    o = assert_bf16_outputs(g_out, hl.out, res["out_exact"], out_m & written_bf16(hl.out), what=f"layer {l} out")
    c = assert_f32_close(g_corr, res["corr_exact"], corr_m, what=f"layer {l} corr")
    if stats is not None:
        stats.append((l, o, c))


def check_commit_layer(prob, l, hl, exact, meta, before=None, mask=None):
    """GPU committed state of layer l vs the oracle's exact fold.  Items that
    commit nothing must keep the GPU's own pre-commit state bit for bit
    (``before[s, h]``; by default the oracle's copy, valid on a first step)."""
    before = hl.state if before is None else before
    cfg = prob.cfg
    H = cfg.H
    lens = np.minimum(np.diff(meta.query_start_loc), cfg.Q)
    acc = np.minimum(np.maximum(meta.num_accepted, 0), lens)
    g_vals, e_vals = [], []
    for b in range(cfg.B):
        s = int(meta.state_indices[b])
        for h in range(H):
            if mask is not None and not mask[b * H + h]:
                continue
            if s <= 0:
                continue
            gs = prob.state[l, s, h].cpu().numpy()
            if acc[b] == 0:
                np.testing.assert_array_equal(gs, before[s, h], err_msg="commit of 0 tokens changed the state")
                continue
            g_vals.append(gs)
            e_vals.append(exact[b, h])
    if g_vals:
        g = np.stack(g_vals)
        e = np.stack(e_vals)
        return assert_f32_close(g, e, np.ones(g.shape, bool), what=f"layer {l} committed state")
    return None


def run_and_check(prob, *, commit=True, mask=None, layers=None, variant="auto", workspace=None):
    """Verify every layer on the GPU, then (optionally) commit all layers in one
    launch; compare each with the oracle run on host copies of the inputs.
    ``workspace``: the device workspace to use (error bits zero), else a new one."""
    cfg = prob.cfg
    meta = prob.meta
    layers = list(range(cfg.L)) if layers is None else layers
    for t in (prob.out, prob.corr, prob.key_gate):
        canary_fill_(t)
    live = meta.state_indices[meta.state_indices > 0]
    hls = {l: host_layer(prob, l, slots=live if mask is not None else None) for l in layers}
    ws = kda.new_workspace(DEV) if workspace is None else workspace
    dm = device_meta(meta, DEV)
    for l in range(cfg.L):
        verify_layer(prob, l, dm, workspace=ws, variant=variant)
    assert kda.read_device_error(ws) == 0
    stats = []
    for l in layers:
        hl = hls[l]
        state_host = hl.state.copy()
        res = run_verify(prob, hl, want_exact=True, item_mask=mask)
        check_verify_layer(prob, l, hl, res, meta, mask=mask, stats=stats)
        # the verify never writes the checkpoint
        idx = np.unique(live).astype(np.int64)
        g_state = prob.state[l][torch.as_tensor(idx, device=DEV)].cpu().numpy()
        np.testing.assert_array_equal(g_state, state_host[idx], err_msg="verify modified the state")
    if commit:
        ctx = commit_context(prob)
        commit_all(ctx, dm, workspace=ws)
        assert kda.read_device_error(ws) == 0
        for l in layers:
            hl = hls[l]
            exact = run_commit(prob, hl, want_exact=True, item_mask=mask)
            check_commit_layer(prob, l, hl, exact, meta, mask=mask)
    return stats


# --------------------------------------------------------------------------- small, every element

C0_VARIANTS = {
    "default": {},
    "lower_bound": dict(lower_bound=-5.0),
    "seq_first": dict(conv_dim_first=False),
    "fp32_weight": dict(conv_weight_fp32=True),
    "no_conv_offsets": dict(conv_offsets=False),
    "record_rows": dict(record_by_request=True),
    "null_slot": dict(null_count=1),
    "window3": dict(Q=3),
    "window2": dict(Q=2),
    "window1": dict(Q=1),
    # windows of 5 to 7 run the window-of-8 build with the scratch laid out
    # for their own Q (the inputs warp then copies the block in parts)
    "window6": dict(Q=6),
}


@pytest.mark.parametrize("variant", sorted(C0_VARIANTS))
def test_c0_tiny(variant):
    prob = make_problem(CONFIGS["C0"].replace(**C0_VARIANTS[variant]), DEV)
    run_and_check(prob)


def test_c1_decode_verify_full_size():
    prob = make_problem(CONFIGS["C1"], DEV)
    assert (prob.meta.state_indices <= 0).sum() == 4
    run_and_check(prob)


def test_c2_verify_then_commit_reduced():
    prob = make_problem(CONFIGS["C2"], DEV, B=40, L=3, slots=64)
    run_and_check(prob)


def test_c3_long_window_reduced():
    prob = make_problem(CONFIGS["C3"], DEV, B=48, slots=128)
    run_and_check(prob)


def test_c4_deferred_chain_reduced():
    """Three decode steps: commit the previous step's pending tokens (all
    layers, one launch), then verify every layer with the conv offset set to
    those same pending counts.  Odd token rows are 8-byte aligned only."""
    prob = make_problem(CONFIGS["C4"], DEV, B=96, L=2, slots=256)
    cfg = prob.cfg
    assert fused_rows_misaligned(prob)
    rng = np.random.default_rng(123)
    ctx = commit_context(prob)
    hls = [host_layer(prob, l) for l in range(cfg.L)]
    meta_prev = None
    ws = kda.new_workspace(DEV)
    for step in range(3):
        meta = prob.meta if step == 0 else next_step_metadata(prob, rng)
        if step > 0:
            dm_prev = device_meta(meta_prev, DEV)
            gpu_before = prob.state.cpu().numpy()
            commit_all(ctx, dm_prev, workspace=ws)
            for l in range(cfg.L):
                exact = run_commit(prob, hls[l], meta=meta_prev, want_exact=True)
                check_commit_layer(prob, l, hls[l], exact, meta_prev, before=gpu_before[l])
            # new activations for the step
            g = torch.Generator(device=DEV).manual_seed(1000 + step)
            prob.fused = (torch.randn((cfg.L, meta.T, prob.fused.shape[2]), generator=g, device=DEV)
                          ).to(torch.bfloat16)
            prob.out = torch.empty((cfg.L, meta.T, cfg.H * cfg.K), dtype=torch.bfloat16, device=DEV)
            for l in range(cfg.L):
                hls[l].fused = to_bits(prob.fused[l])
                hls[l].out = np.empty((meta.T, cfg.H * cfg.K), np.uint16)
        prob.meta = meta
        for t in (prob.out, prob.corr, prob.key_gate):
            canary_fill_(t)
        for l in range(cfg.L):
            hls[l].out[...] = 0x7FA5
            hls[l].corr.view(np.uint32)[...] = 0x7FC0DEAD
            hls[l].key_gate[...] = 0x7FA5
        dm = device_meta(meta, DEV)
        for l in range(cfg.L):
            verify_layer(prob, l, dm, workspace=ws)
        assert kda.read_device_error(ws) == 0
        for l in range(cfg.L):
            res = run_verify(prob, hls[l], meta=meta, want_exact=True)
            check_verify_layer(prob, l, hls[l], res, meta)
        meta_prev = meta


def fused_rows_misaligned(prob):
    row_bytes = prob.fused.stride(1) * 2
    return row_bytes % 16 == 8


def test_activation_rows_at_odd_element_offsets():
    """Projection rows that start 2 bytes past a 16-byte boundary."""
    cfg = CONFIGS["C0"]
    prob = make_problem(cfg, DEV)
    wide = torch.zeros((cfg.L, prob.fused.shape[1], prob.fused.shape[2] + 1), dtype=torch.bfloat16, device=DEV)
    wide[:, :, 1:] = prob.fused
    prob.fused = wide[:, :, 1:]
    assert prob.fused.data_ptr() % 16 == 2
    for t in (prob.out, prob.corr, prob.key_gate):
        canary_fill_(t)
    hl = host_layer(prob, 0)
    hl.fused = np.ascontiguousarray(to_bits(prob.fused[0]))
    dm = device_meta(prob.meta, DEV)
    verify_layer(prob, 0, dm)
    res = run_verify(prob, hl, want_exact=True)
    check_verify_layer(prob, 0, hl, res, prob.meta)


# --------------------------------------------------------------------------- full sizes, sampled

@pytest.mark.parametrize("name,layers,items", [("C2", [0, 11, 23], 48), ("C3", [0], 96), ("C4", [0, 11], 64)])
def test_full_size_sampled(name, layers, items):
    """The full benchmark workload in the benchmark's launch configuration
    (every layer verified, one commit launch over all layers); the oracle
    recomputes a random sample of (request, head) items."""
    prob = make_problem(CONFIGS[name], DEV)
    mask = _item_mask(prob, items, seed=7)
    run_and_check(prob, mask=mask, layers=layers)


# --------------------------------------------------------------------------- invariants on the GPU

def test_commit_prefix_property_on_gpu():
    """GPU commit of m tokens equals the oracle verify's running state after m."""
    cfg = CONFIGS["C0"].replace(B=6, slots=12)
    for m in range(1, cfg.Q + 1):
        prob = make_problem(cfg, DEV)
        prob.meta.num_accepted = np.full(cfg.B, m, np.int32)
        hl = host_layer(prob, 0)
        res = run_verify(prob, hl, want_running=True)
        dm = device_meta(prob.meta, DEV)
        verify_layer(prob, 0, dm)
        commit_all(commit_context(prob), dm)
        lens = np.minimum(np.diff(prob.meta.query_start_loc), cfg.Q)
        for b in range(cfg.B):
            s = int(prob.meta.state_indices[b])
            mm = min(m, int(lens[b]))
            got = prob.state[0, s].cpu().numpy()
            ref = res["running_state"][b, :, mm - 1]
            assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max()


def test_verify_and_commit_are_bitwise_reproducible():
    """Two runs on the same inputs write the same bits (no order-dependent
    floating-point reductions across warps or CTAs)."""
    runs = []
    for _ in range(2):
        p2 = make_problem(CONFIGS["C2"], DEV, B=48, L=2, slots=96)
        dm = device_meta(p2.meta, DEV)
        for l in range(p2.cfg.L):
            verify_layer(p2, l, dm)
        commit_all(commit_context(p2), dm)
        torch.cuda.synchronize()
        runs.append([t.view(torch.int16 if t.element_size() == 2 else torch.int32).cpu().numpy()
                     for t in (p2.out, p2.corr, p2.key_gate, p2.conv_state, p2.state)])
    for a, b in zip(*runs):
        np.testing.assert_array_equal(a, b)


def test_empty_and_all_null_batches():
    cfg = CONFIGS["C0"]
    prob = make_problem(cfg, DEV)
    dm = device_meta(prob.meta, DEV)
    # zero tokens: a no-op
    empty_qsl = torch.zeros(cfg.B + 1, dtype=torch.int32, device=DEV)
    before = prob.conv_state.clone()
    kda.verify(mixed_qkv=prob.fused[0, :0, : 3 * cfg.H * cfg.K], raw_gate=prob.fused[0, :0, 768:1024],
               raw_beta=prob.fused[0, :0, 1024:1028], A_log=prob.A_log[0], dt_bias=prob.dt_bias[0],
               lower_bound=None, state=prob.state[0], correction=prob.corr[0], key_gate=prob.key_gate[0],
               query_start_loc=empty_qsl, state_indices=dm.state_indices, conv_state=prob.conv_state[0],
               conv_weight=prob.conv_weight[0], out=prob.out[0, :0], window=cfg.Q)
    torch.cuda.synchronize()
    assert torch.equal(before, prob.conv_state)
    # every request null: zero outputs only
    prob.meta.state_indices[:] = [0, -1, 0, -3]
    run_and_check(prob)
    assert (to_bits(prob.out[0]) == 0).all()


def test_zero_length_requests_and_long_queries():
    """query_len 0 (repeated query_start_loc) writes nothing; query_len > Q
    verifies the first Q tokens only."""
    cfg = CONFIGS["C0"].replace(B=4, slots=8)
    prob = make_problem(cfg, DEV)
    T = prob.meta.T
    qsl = np.array([0, 0, min(T, 6), min(T, 6), T], np.int32)  # requests 0 and 2 empty, 1 maybe > Q
    prob.meta.query_start_loc = qsl
    run_and_check(prob)


def test_device_errors_skip_only_the_bad_items():
    cfg = CONFIGS["C0"].replace(B=4, slots=8)
    prob = make_problem(cfg, DEV)
    prob.meta.state_indices[1] = 99  # beyond the pool
    ws = kda.new_workspace(DEV)
    dm = device_meta(prob.meta, DEV)
    canary_fill_(prob.out)
    verify_layer(prob, 0, dm, workspace=ws)
    flags = kda.read_device_error(ws)
    assert flags & kda.DEVERR_SLOT_RANGE
    out = to_bits(prob.out[0])
    bos, eos = int(prob.meta.query_start_loc[1]), int(prob.meta.query_start_loc[2])
    assert (out[bos:eos] == 0x7FA5).all()
    assert (out[:bos] != 0x7FA5).all() and (out[eos:] != 0x7FA5).all()
    # a record row out of range
    prob2 = make_problem(cfg.replace(record_by_request=True), DEV)
    prob2.meta.record_indices[2] = 4
    ws2 = kda.new_workspace(DEV)
    verify_layer(prob2, 0, device_meta(prob2.meta, DEV), workspace=ws2)
    assert kda.read_device_error(ws2) & kda.DEVERR_ROW_RANGE
    # a decreasing query_start_loc
    prob3 = make_problem(cfg, DEV)
    q = prob3.meta.query_start_loc.copy()
    q[2] = q[1] - 1 if q[1] > 0 else q[1]
    prob3.meta.query_start_loc = q
    ws3 = kda.new_workspace(DEV)
    verify_layer(prob3, 0, device_meta(prob3.meta, DEV), workspace=ws3)
    commit_all(commit_context(prob3), device_meta(prob3.meta, DEV), workspace=ws3)
    assert kda.read_device_error(ws3) & kda.DEVERR_TOKEN_RANGE
