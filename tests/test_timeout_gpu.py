"""The verify kernel's bounded device waits, made to run out through
kda_verify_debug: one item's inputs are withheld (its slot never fills), and
with a 1 ms limit the wait for it gives up.  The test checks that the
kernel returns, that KDA_DEVERR_TIMEOUT is reported, that every item is
either verified as the oracle says or left untouched (the withheld one and
at most a few others that the stopped CTA had drawn), and that the context
and the workspace's ticket counter stay usable for a plain verify afterwards.  No GPU fault is involved: the kernel
only stops waiting.  The same entry point's timing hook (each CTA's start and
finish on the global timer) is checked to cover the launch and to leave the
outputs unchanged."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_ssm_kda_gb300 as kda
from compare import written_bf16, written_f32
from linear_attention_ssm_kda_gb300 import _build
from oracle_io import host_layer, run_verify
from test_parity_gpu import _masks_for_items, check_verify_layer, run_and_check
from workloads import CONFIGS, canary_fill_, make_problem, to_bits
from workloads.drive import device_meta, verify_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    kda.load_library()


def _item_windows(prob, meta):
    """Per item (b H + h): its token rows (bos, n), n clipped to the window."""
    cfg = prob.cfg
    qsl = np.asarray(meta.query_start_loc)
    bos = np.repeat(qsl[:-1], cfg.H)
    n = np.clip(np.repeat(qsl[1:] - qsl[:-1], cfg.H), 0, cfg.Q)
    return bos, n


def test_withheld_item_times_out_and_the_rest_is_verified():
    prob = make_problem(CONFIGS["C2"], DEV, B=40, L=1, slots=64)
    cfg, meta = prob.cfg, prob.meta
    H, K = cfg.H, cfg.K
    items = cfg.B * H
    grid = min(items, torch.cuda.get_device_properties(0).multi_processor_count)
    assert items > 3 * grid
    bos, n = _item_windows(prob, meta)
    withhold = int(np.flatnonzero((np.arange(items) >= 2 * grid) & (n > 0))[0])
    for t in (prob.out, prob.corr, prob.key_gate):
        canary_fill_(t)
    hl = host_layer(prob, 0)
    ws = kda.new_workspace(DEV)
    dm = device_meta(meta, DEV)
    verify_layer(prob, 0, dm, workspace=ws, debug=(withhold, 1_000_000))
    torch.cuda.synchronize()
    flags = kda.read_device_error(ws)
    assert flags & kda.DEVERR_TIMEOUT, f"device error bits 0x{flags:x}"
    assert flags & ~kda.DEVERR_TIMEOUT == 0

    # Items are dealt at run time, so which items the stopped CTA held is not
    # fixed: every item with a window is either verified (all its output rows
    # written) or untouched, the withheld one is untouched, and the stopped
    # CTA held at most a few more (its lead of drawn items: 3 past the one in
    # hand plus a batch of at most 8).
    written = written_bf16(to_bits(prob.out[0]))
    stopped = np.zeros(items, bool)
    for it in np.flatnonzero(n > 0):
        b, h = divmod(int(it), H)
        w = written[bos[it]: bos[it] + n[it], h * K:(h + 1) * K]
        assert w.all() or not w.any(), f"item {it} half written"
        stopped[it] = not w.any()
    assert stopped[withhold]
    assert stopped.sum() <= 12, np.flatnonzero(stopped)
    res = run_verify(prob, hl, want_exact=True)
    check_verify_layer(prob, 0, hl, res, meta, mask=(~stopped).astype(np.uint8))
    out_m, rec_m, _ = _masks_for_items(prob, meta, stopped.astype(np.uint8))
    assert out_m.any() and rec_m.any()
    assert not written_f32(prob.corr[0].cpu().numpy())[rec_m].any()
    assert not written_bf16(to_bits(prob.key_gate[0]))[rec_m].any()

    # the ticket counter is back at zero: a plain verify afterwards, with the
    # same workspace (error words cleared), covers every item
    ws[:2].zero_()
    run_and_check(make_problem(CONFIGS["C2"], DEV, B=40, L=1, slots=64, seed=5), workspace=ws)


def test_context_usable_after_a_timeout():
    prob = make_problem(CONFIGS["C0"], DEV)
    ws = kda.new_workspace(DEV)
    verify_layer(prob, 0, device_meta(prob.meta, DEV), workspace=ws, debug=(1, 1_000_000))
    assert kda.read_device_error(ws) & kda.DEVERR_TIMEOUT
    run_and_check(make_problem(CONFIGS["C0"], DEV, seed=11))


@pytest.mark.parametrize("variant", ["cuda_core", "tcgen05"])
def test_cta_times_cover_the_launch_and_change_nothing(variant):
    """The timing hook of kda_verify_debug: every CTA of the launch records a
    start no later than its finish, entries past the grid stay as they were,
    and the outputs are those of the plain verify, bit for bit."""
    prob = make_problem(CONFIGS["C2"], DEV, B=40, L=1, slots=64)
    cfg = prob.cfg
    items = cfg.B * cfg.H
    grid = min(items, torch.cuda.get_device_properties(0).multi_processor_count)
    dm = device_meta(prob.meta, DEV)
    conv0 = prob.conv_state.clone()
    ws = kda.new_workspace(DEV)
    verify_layer(prob, 0, dm, workspace=ws, variant=variant)
    plain = [t.clone() for t in (prob.out, prob.corr, prob.key_gate, prob.conv_state)]
    prob.conv_state.copy_(conv0)
    times = torch.full((2 * items,), -1, dtype=torch.int64, device=DEV)
    verify_layer(prob, 0, dm, workspace=ws, variant=variant, debug=(-1, 1_000_000_000, times))
    torch.cuda.synchronize()
    assert kda.read_device_error(ws) == 0
    for a, b in zip(plain, (prob.out, prob.corr, prob.key_gate, prob.conv_state)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    t = times.cpu().numpy().reshape(-1, 2)
    assert (t[:grid] > 0).all() and (t[:grid, 0] <= t[:grid, 1]).all()
    assert (t[grid:] == -1).all()
    span = t[:grid, 1].max() - t[:grid, 0].min()
    assert 0 < span < 1_000_000_000
