"""The verify kernel's bounded device waits, made to run out through
kda_verify_debug: one item's inputs are withheld (its slot never fills), and
with a 1 ms limit the wait for it gives up.  The test checks that the
kernel returns, that KDA_DEVERR_TIMEOUT is reported, that the items of the
other CTAs and the owning CTA's earlier items match the oracle, that the
owning CTA's later items are left unwritten, and that the context stays
usable for a plain verify afterwards.  No GPU fault is involved: the kernel
only stops waiting."""
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


def test_withheld_item_times_out_and_the_rest_is_verified():
    prob = make_problem(CONFIGS["C2"], DEV, B=40, L=1, slots=64)
    cfg, meta = prob.cfg, prob.meta
    items = cfg.B * cfg.H
    grid = min(items, torch.cuda.get_device_properties(0).multi_processor_count)
    assert items > 3 * grid
    withhold = 2 * grid  # the third item of the first CTA
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

    it = np.arange(items)
    stopped = (it % grid == 0) & (it // grid >= 2)  # the first CTA, from the withheld item on
    res = run_verify(prob, hl, want_exact=True)
    check_verify_layer(prob, 0, hl, res, meta, mask=(~stopped).astype(np.uint8))
    out_m, rec_m, _ = _masks_for_items(prob, meta, stopped.astype(np.uint8))
    assert out_m.any() and rec_m.any()
    assert not written_bf16(to_bits(prob.out[0]))[out_m].any()
    assert not written_f32(prob.corr[0].cpu().numpy())[rec_m].any()
    assert not written_bf16(to_bits(prob.key_gate[0]))[rec_m].any()


def test_context_usable_after_a_timeout():
    prob = make_problem(CONFIGS["C0"], DEV)
    ws = kda.new_workspace(DEV)
    verify_layer(prob, 0, device_meta(prob.meta, DEV), workspace=ws, debug=(1, 1_000_000))
    assert kda.read_device_error(ws) & kda.DEVERR_TIMEOUT
    run_and_check(make_problem(CONFIGS["C0"], DEV, seed=11))
