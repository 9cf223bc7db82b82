"""The tensor-core verify (K = 128; the default for windows of 8, forced here
for every window with the "tcgen05" variant: P | R from tcgen05 tf32 MMAs with
a hi/lo split of the state) against the oracle, under the same comparison
rules as the CUDA-core path."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_ssm_kda_gb300 as kda
from linear_attention_ssm_kda_gb300 import _build
from test_parity_gpu import run_and_check
from workloads import CONFIGS, make_problem
from workloads.drive import device_meta, verify_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _lib():
    _build.build()
    kda.load_library()


def test_c1_full_size_with_null_slots():
    prob = make_problem(CONFIGS["C1"], DEV)
    assert (prob.meta.state_indices <= 0).sum() == 4
    run_and_check(prob, variant="tcgen05")


def test_c2_verify_then_commit_reduced():
    prob = make_problem(CONFIGS["C2"], DEV, B=40, L=3, slots=64)
    run_and_check(prob, variant="tcgen05")


def test_c3_window_of_eight_reduced():
    """Q = 8: the MMA's N is 32 (16 vectors' hi and lo rows)."""
    prob = make_problem(CONFIGS["C3"], DEV, B=48, slots=128)
    run_and_check(prob, variant="tcgen05")


def test_c3_cuda_core_path_when_forced():
    """The "cuda_core" variant keeps the CUDA-core gemv for windows of 8."""
    prob = make_problem(CONFIGS["C3"], DEV, B=48, slots=128)
    run_and_check(prob, variant="cuda_core")


@pytest.mark.parametrize("window", [2, 5, 7])
@pytest.mark.parametrize("variant", ["tcgen05", "cuda_core"])
def test_windows_below_the_build_maximum(window, variant):
    """Windows of 2 and of 5 to 7 run the builds for 4 and 8 with a smaller
    Q: the MMA's B operand is zero past 2n, and the scratch is laid out for
    the call's own Q."""
    prob = make_problem(CONFIGS["C3"].replace(Q=window), DEV, B=32, slots=96)
    run_and_check(prob, variant=variant)


def test_c4_null_slots_and_misaligned_rows_reduced():
    prob = make_problem(CONFIGS["C4"], DEV, B=96, L=2, slots=256)
    assert (prob.meta.state_indices <= 0).sum() > 0
    run_and_check(prob, variant="tcgen05")


def test_differs_from_the_cuda_core_path_only_by_rounding():
    """Both instantiations run on the same inputs; the outputs agree to the
    verify tolerance but not bit for bit, so the tensor-core kernel did run."""
    got = {}
    for variant in ("tcgen05", "cuda_core"):
        prob = make_problem(CONFIGS["C2"], DEV, B=48, L=1, slots=96)
        dm = device_meta(prob.meta, DEV)
        verify_layer(prob, 0, dm, variant=variant)
        torch.cuda.synchronize()
        got[variant] = prob.corr[0].cpu().numpy()
    a, b = got["tcgen05"], got["cuda_core"]
    live = np.isfinite(a) & np.isfinite(b)
    assert not np.array_equal(a[live].view(np.uint32), b[live].view(np.uint32))
    assert np.abs(a[live] - b[live]).max() <= 1e-4 * np.abs(b[live]).max()
