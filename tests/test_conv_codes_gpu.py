"""The conv pass's bf16 codes where the decision is hard, bit for bit: the
rows of tests/golden/conv_adversarial.txt (SiLU next to a rounding boundary,
tap sums exactly on a bf16 midpoint, |y| beyond the fp32 range of e^-|y|)
as fp32 conv weights of the key channels, fed with inputs of 1.0, so that
every token of every window has the row's sum.  The key records carry the
codes; the expected ones come from the oracle, whose codes for these rows the
CPU pins check against an arbitrary-precision evaluation."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_ssm_kda_gb300 as kda
import oracle
from compare import conv_adversarial_rows
from linear_attention_ssm_kda_gb300 import _build
from workloads import CONFIGS, make_problem, to_bits
from workloads.drive import device_meta, verify_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    kda.load_library()


@pytest.mark.parametrize("dim_first", [False, True])
def test_conv_codes_on_adversarial_rows(dim_first):
    cfg = CONFIGS["C1"].replace(conv_weight_fp32=True, conv_dim_first=dim_first)
    prob = make_problem(cfg, DEV, B=6, slots=16)
    cfg = prob.cfg
    H, K = cfg.H, cfg.K
    HK = H * K
    kinds, rows = conv_adversarial_rows()
    nrow = rows.shape[0]
    assert nrow <= HK
    # key channels c < nrow take the rows; inputs of 1.0 on every key channel
    prob.conv_weight[0, HK:HK + nrow] = torch.tensor(rows, dtype=torch.float32, device=DEV)
    prob.fused[0, :, HK:2 * HK] = 1.0
    if dim_first:   # [slots, 3HK, taps]
        prob.conv_state[0, :, HK:2 * HK, :] = 1.0
    else:           # [slots, taps, 3HK]
        prob.conv_state[0, :, :, HK:2 * HK] = 1.0
    ws = kda.new_workspace(DEV)
    verify_layer(prob, 0, device_meta(prob.meta, DEV), workspace=ws)
    assert kda.read_device_error(ws) == 0
    want = oracle.conv_silu_bf16(rows, np.ones_like(rows))
    meta = prob.meta
    kg = to_bits(prob.key_gate[0])          # [rows, H, Q, 2K]
    checked = 0
    for b in range(cfg.B):
        s = int(meta.state_indices[b])
        n = min(int(meta.query_start_loc[b + 1] - meta.query_start_loc[b]), cfg.Q)
        if s <= 0 or n <= 0:
            continue
        r = s if meta.record_indices is None else int(meta.record_indices[b])
        for t in range(n):
            got = kg[r, :, t, :K].reshape(HK)[:nrow]
            bad = np.flatnonzero(got != want)
            assert bad.size == 0, (f"request {b} token {t}: {bad.size} codes differ, rows {bad[:4]} "
                                   f"({kinds[bad[:4]]}): got {got[bad[:4]]}, want {want[bad[:4]]}")
            checked += 1
    assert checked >= 4
