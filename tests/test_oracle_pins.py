"""Pins of the CPU oracle to things other than itself: hand-worked golden
values, library routines, closed forms, invariants of the delta rule, and an
independent matrix-form brute force at K = V = 4.  CPU only."""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit

import brute
import compare
import oracle
from oracle_io import host_layer, run_commit, run_verify
from workloads import CONFIGS, Config, make_problem

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# --------------------------------------------------------------------------- scalars

def test_bf16_round_golden():
    for x, bits, *_ in _golden_rows("bf16_round.txt"):
        assert oracle.bf16_round(float.fromhex(x)) == int(bits, 16), x


def test_bf16_round_matches_torch_on_fp32_values():
    # torch rounds fp32 -> bf16 to nearest even; for values exactly representable
    # in fp32, rounding straight from double must agree.
    g = torch.Generator().manual_seed(7)
    x = torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 8)
    x = torch.cat([x, torch.tensor([0.0, -0.0, 1e-40, -3e-39, 3.3e38, -3.39e38])])
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_round(float(v)) for v in x.numpy()], np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_gate_golden_points():
    for raw_g, dt, A, lb, expected, *_ in _golden_rows("gate_points.txt"):
        lbv = None if lb == "none" else float(lb)
        got = oracle.gate(float(raw_g), float(dt), float(A), lbv)
        exp_v = float(expected)
        assert got == pytest.approx(exp_v, rel=1e-15, abs=0.0), (raw_g, dt, A, lb)
        assert math.copysign(1.0, got) == math.copysign(1.0, exp_v)


def test_gate_against_library_routines():
    rng = np.random.default_rng(3)
    for _ in range(500):
        u = rng.normal(0, 8)
        A = math.exp(rng.uniform(-1, 1))
        sp = u if u > 20 else np.logaddexp(0.0, u)
        # log(1 + e^u) (the pages' form) loses relative accuracy once e^u is below
        # the double epsilon; its absolute error stays at the 1e-16 level
        assert oracle.gate(u, 0.0, A) == pytest.approx(-A * sp, rel=1e-13, abs=1e-15)
        assert oracle.gate(u, 0.0, A, -5.0) == pytest.approx(-5.0 * expit(A * u), rel=1e-13)
    # the threshold switch at 20 is continuous to ~e^-20
    assert abs(oracle.gate(20.0 + 1e-9, 0, 1) - oracle.gate(20.0 - 1e-9, 0, 1)) < 1e-8


def _bf16_bits(v):
    """bf16 codes (RNE) of float values via torch."""
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("fp32_weights", [False, True])
def test_conv_code_is_the_correct_rounding(fp32_weights):
    """Codes of conv + SiLU on random taps equal the correctly rounded exact
    value: double decides where it is unambiguous, 60 digits elsewhere."""
    rng = np.random.default_rng(7 + fp32_weights)
    n, W = 200_000, 4
    gen = torch.Generator().manual_seed(17 + fp32_weights)
    x = brute.bf16_values(_bf16_bits(torch.randn(n, W, dtype=torch.float32, generator=gen).mul_(1.5).numpy()))
    w = rng.normal(0, 0.5, (n, W)).astype(np.float32).astype(np.float64)
    if not fp32_weights:
        w = brute.bf16_values(_bf16_bits(w))
    codes = oracle.conv_silu_bf16(w, x)
    y = (w * x).sum(axis=1)
    brute.assert_codes_exact(codes, y)
    # unit taps pick one input: y is that bf16 value exactly
    onehot = np.eye(W)
    got = oracle.conv_silu_bf16(onehot, x[:W])
    brute.assert_codes_exact(got, np.diag(x[:W]))


def _near_boundary_inputs(count, seed, lo_exp=-45, hi_exp=-30):
    """Conv inputs whose SiLU lies a chosen distance from a bf16 rounding
    boundary m: SiLU(y*) = m (1 + d) with |d| = 2^-u, u uniform in
    (-hi_exp, -lo_exp), solved for y* in 60 digits; y* is split into four fp32
    pieces (the weights, each times an input 1.0), whose sum is y* to about
    2^-96.  Returns (w, x, d, lower): lower is the bf16 code on the near-zero
    side of m, so the correct code is lower + 1 exactly when d > 0."""
    import mpmath
    rng = np.random.default_rng(seed)
    ws, ds, lows = [], [], []
    with mpmath.workdps(60):
        for _ in range(count):
            if rng.random() < 0.7:       # positive branch, SiLU from 1e-3 to 40
                target = float(np.exp(rng.uniform(np.log(1e-3), np.log(40.0))))
                lo, hi = 0.0, 60.0
            else:                        # negative values on the branch y in (-1.278, 0)
                target = -float(np.exp(rng.uniform(np.log(1e-3), np.log(0.27))))
                lo, hi = -1.2784645, 0.0
            code = int(_bf16_bits(np.array([target]))[0])
            mid = (brute.bf16_values(np.array([code], np.uint16))[0]
                   + brute.bf16_values(np.array([code + 1], np.uint16))[0]) / 2
            d = float(rng.choice([-1.0, 1.0]) * 2.0 ** -rng.uniform(-hi_exp, -lo_exp))
            goal = mpmath.mpf(mid) * (1 + mpmath.mpf(d))
            f = lambda yy: yy / (1 + mpmath.exp(-yy)) - goal  # noqa: E731
            r = mpmath.findroot(f, (mpmath.mpf(lo) + 1e-30, mpmath.mpf(hi)), solver="bisect", tol=1e-55)
            pieces = []
            for _ in range(4):
                p = float(np.float32(float(r)))
                pieces.append(p)
                r = r - p
            ws.append(pieces)
            ds.append(d)
            lows.append(code)
    return np.array(ws), np.ones((count, 4)), np.array(ds), np.array(lows, np.uint16)


def test_conv_code_next_to_rounding_boundaries():
    """Adversarial pin: SiLU values placed 2^-45 .. 2^-30 (relative) from a
    bf16 rounding boundary, where a plain fp32 evaluation picks the wrong
    neighbour about half the time and double precision still decides.  The
    oracle's codes must be the exact ones."""
    pytest.importorskip("mpmath")
    w, x, d, lower = _near_boundary_inputs(600, seed=23)
    codes = oracle.conv_silu_bf16(w, x)
    want = brute.silu_codes_exact(w * x)
    np.testing.assert_array_equal(codes, want)
    # the 60-digit reference lands on the side of the boundary the construction chose
    np.testing.assert_array_equal(want, lower + (d > 0).astype(np.uint16))
    # the inputs are sharp: fp32 arithmetic gets a good share of them wrong
    yf = (w * x).sum(axis=1).astype(np.float32)
    naive = _bf16_bits(yf / (np.float32(1) + np.exp(-yf)))
    assert np.mean(naive != want) > 0.1


def _large_midpoint_sums(seed):
    """Conv inputs whose tap sum y is exactly a bf16 midpoint above 37, where
    double precision cannot tell SiLU(y) = y - y e^-y / (1 + e^-y) from y: one
    tap w x with w = 1.5 2^a and x = v 2^b (both bf16), 3 v a 9-bit odd
    number, the other taps zero.  Returns (w, x, y, n3): n3 marks the sums
    whose even neighbour is the upper one, where nearest-even rounding of y
    gives the wrong code."""
    rng = np.random.default_rng(seed)
    ws, xs, ys, n3 = [], [], [], []
    for v in range(87, 171, 2):             # 3 v in [261, 511]: nine significant bits, the last one set
        sh = int(rng.integers(-2, 6))       # y = 3 v 2^sh, from about 65 to 16 000
        a = int(rng.integers(-2, 3))        # the power of two split between w and x
        w = 1.5 * 2.0 ** a
        x = v * 2.0 ** (sh - a + 1)         # w x = 3 v 2^sh
        y = w * x
        ws.append([0.0, 0.0, 0.0, w])
        xs.append([0.0, 0.0, 0.0, x])
        ys.append(y)
        n3.append((3 * v) % 4 == 3)
    return np.array(ws), np.array(xs), np.array(ys), np.array(n3)


def test_conv_code_large_sums_on_a_midpoint():
    """A sum that is exactly a bf16 midpoint stands for SiLU just below it:
    the code is the one nearer zero (the exact evaluation decides), although
    double precision sees SiLU(y) == y there and nearest-even would pick the
    upper code in about half of the cases."""
    pytest.importorskip("mpmath")
    w, x, y, n3 = _large_midpoint_sums(seed=31)
    assert (y > 37).all() and (brute.bf16_midpoint_distance(y) == 0).all()
    want = brute.silu_codes_exact(w * x)
    np.testing.assert_array_equal(oracle.conv_silu_bf16(w, x), want)
    np.testing.assert_array_equal(want, brute.bf16_rne(y - y * 2.0 ** -30))  # the code below the midpoint
    assert (want != brute.bf16_rne(y))[n3].all() and n3.sum() >= 10
    # negative sums of the same size: SiLU is tiny there, and decided plainly
    np.testing.assert_array_equal(oracle.conv_silu_bf16(w, -x), brute.silu_codes_exact(w * -x))


def test_conv_adversarial_fixture_codes_are_exact():
    """The adversarial rows the GPU conv test runs (tests/golden/
    conv_adversarial.txt): the oracle's codes are the exact ones."""
    pytest.importorskip("mpmath")
    kinds, w = compare.conv_adversarial_rows()
    assert set(kinds) == {"near", "tie", "large"} and len(w) > 500
    np.testing.assert_array_equal(oracle.conv_silu_bf16(w, np.ones_like(w)), brute.silu_codes_exact(w))


def test_silu_codes_exact_against_known_roundings():
    """The 60-digit reference itself: SiLU(0) = 0, large y rounds like y, and
    values far from a boundary agree with the double evaluation."""
    assert int(brute.silu_codes_exact([0.0])[0]) == 0
    big = np.array([64.0, 100.0, 3.0e4])
    np.testing.assert_array_equal(brute.silu_codes_exact(big), _bf16_bits(big))
    yy = np.linspace(-8, 8, 2001)
    s = yy * expit(yy)
    far = brute.bf16_midpoint_distance(s) > 1e-9
    np.testing.assert_array_equal(brute.silu_codes_exact(yy[far]), brute.bf16_rne(s[far]))
    # the test's own rounding agrees with torch's on fp32-exact values, subnormals included
    f = np.concatenate([s, s * 2.0 ** -130, -s * 2.0 ** -128]).astype(np.float32)
    np.testing.assert_array_equal(brute.bf16_rne(f.astype(np.float64)), _bf16_bits(f))


# --------------------------------------------------------------------------- brute force

def _codes(values):
    """bf16 codes of bf16-exact double values."""
    return (np.asarray(values, np.float64).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _tiny(**kw):
    base = Config("tiny", B=3, H=2, K=4, Q=4, L=1, slots=6, seed=11, state_std=0.3)
    return base.replace(**kw)


def _item_inputs(prob, hl, b, h, meta=None):
    """The test's own reading of the buffers for one (request, head)."""
    cfg = prob.cfg
    meta = meta or prob.meta
    H, K, Q, W = cfg.H, cfg.K, cfg.Q, cfg.W
    HK = H * K
    bos = int(meta.query_start_loc[b])
    n = min(int(meta.query_start_loc[b + 1]) - bos, Q)
    s = int(meta.state_indices[b])
    a = 1 if meta.num_accepted_prev is None else min(max(int(meta.num_accepted_prev[b]), 1), Q)
    chans = np.concatenate([g * HK + h * K + np.arange(K) for g in range(3)])
    cs = hl.conv_state
    if cfg.conv_dim_first:
        hist_bits = cs[s][chans][:, a - 1: a - 1 + W - 1].T
    else:
        hist_bits = cs[s][a - 1: a - 1 + W - 1][:, chans]
    x_bits = hl.fused[bos: bos + n][:, chans]
    w = hl.conv_weight[chans]
    w = w.astype(np.float64) if w.dtype == np.float32 else brute.bf16_values(w)
    raw_g = brute.bf16_values(hl.fused[bos: bos + n, 3 * HK + h * K: 3 * HK + (h + 1) * K])
    raw_beta = brute.bf16_values(hl.fused[bos: bos + n, 4 * HK + h])
    return dict(bos=bos, n=n, s=s, a=a, hist=brute.bf16_values(hist_bits),
                x=brute.bf16_values(x_bits), w=w, raw_g=raw_g, raw_beta=raw_beta,
                S0=hl.state[s, h].astype(np.float64), chans=chans)


@pytest.mark.parametrize("variant", [
    dict(),
    dict(lower_bound=-5.0),
    dict(conv_dim_first=False),
    dict(conv_weight_fp32=True, act_std=2.0),
    dict(conv_offsets=False),
    dict(record_by_request=True, Q=3),
])
def test_verify_matches_matrix_form_bruteforce(variant):
    prob = make_problem(_tiny(**variant))
    cfg = prob.cfg
    hl = host_layer(prob, 0)
    state_before = hl.state.copy()
    res = run_verify(prob, hl, want_exact=True, want_running=True, want_post_conv=True)
    K, H = cfg.K, cfg.H
    meta = prob.meta
    checked = 0
    # re-read the pristine inputs (the oracle updated the conv state in place)
    fresh = host_layer(make_problem(cfg), 0)
    for b in range(cfg.B):
        for h in range(H):
            it = _item_inputs(prob, fresh, b, h)
            if it["n"] <= 0 or it["s"] <= 0:
                continue
            sx, mag, y = brute.conv_silu_exact(it["hist"], it["x"], it["w"])
            post = res["post_conv"][it["bos"]: it["bos"] + it["n"]][:, it["chans"]]
            brute.assert_codes_exact(_codes(post), y)
            q, k, v = post[:, :K], post[:, K: 2 * K], post[:, 2 * K:]
            o, c, states = brute.window(it["S0"], q, k, v, it["raw_g"], it["raw_beta"],
                                        fresh.dt_bias[h * K:(h + 1) * K].astype(np.float64),
                                        float(fresh.A_log[h]), cfg.lower_bound)
            r = it["s"] if meta.record_indices is None else int(meta.record_indices[b])
            n = it["n"]
            np.testing.assert_allclose(res["out_exact"][it["bos"]: it["bos"] + n, h * K:(h + 1) * K],
                                       o, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(res["corr_exact"][r, h, :n], c, rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(res["running_state"][b, h, :n], states, rtol=1e-10, atol=1e-12)
            checked += 1
    assert checked >= 3
    np.testing.assert_array_equal(hl.state, state_before)  # the verify never writes the state


def test_commit_matches_closed_form_fold():
    prob = make_problem(_tiny(B=4, slots=8))
    cfg = prob.cfg
    hl = host_layer(prob, 0)
    run_verify(prob, hl)
    S_before = hl.state.copy()
    exact = run_commit(prob, hl, want_exact=True)
    meta = prob.meta
    K = cfg.K
    folds = 0
    for b in range(cfg.B):
        s = int(meta.state_indices[b])
        n = min(int(meta.query_start_loc[b + 1] - meta.query_start_loc[b]), cfg.Q)
        m = min(max(int(meta.num_accepted[b]), 0), n)
        for h in range(cfg.H):
            if s <= 0 or m == 0:
                continue
            c = hl.corr[s, h, :m].astype(np.float64)
            kg = hl.key_gate[s, h, :m]
            k = brute.bf16_values(kg[:, :K])
            rg = brute.bf16_values(kg[:, K:])
            ref = brute.fold(S_before[s, h].astype(np.float64), c, k, rg,
                             hl.dt_bias[h * K:(h + 1) * K].astype(np.float64),
                             float(hl.A_log[h]), cfg.lower_bound)
            np.testing.assert_allclose(exact[b, h], ref, rtol=1e-10, atol=1e-13)
            np.testing.assert_array_equal(hl.state[s, h], exact[b, h].astype(np.float32))
            folds += 1
    assert folds >= 2


@pytest.mark.parametrize("lb", [None, -5.0])
def test_commit_prefix_property(lb):
    """commit(m) is the verify's running state after m tokens, for every m."""
    cfg = _tiny(B=4, slots=8, K=8, lower_bound=lb)
    prob = make_problem(cfg)
    meta = prob.meta
    hl = host_layer(prob, 0)
    res = run_verify(prob, hl, want_running=True)
    lens = np.minimum(np.diff(meta.query_start_loc), cfg.Q)
    for m in range(0, cfg.Q + 1):
        hl2 = host_layer(prob, 0)
        hl2.corr[...] = hl.corr
        hl2.key_gate[...] = hl.key_gate
        meta.num_accepted = np.full(cfg.B, m, np.int32)
        run_commit(prob, hl2)
        for b in range(cfg.B):
            s = int(meta.state_indices[b])
            mm = min(m, int(lens[b]))
            for h in range(cfg.H):
                if mm == 0:
                    np.testing.assert_array_equal(hl2.state[s, h], hl.state[s, h])
                else:
                    ref = res["running_state"][b, h, mm - 1]
                    # the commit replays fp32-rounded corrections: ~1e-7 relative
                    np.testing.assert_allclose(hl2.state[s, h], ref, rtol=0,
                                               atol=2e-6 * np.abs(ref).max())


@pytest.mark.parametrize("lb", [None, -5.0])
def test_align_commit_boundary_is_the_state_after_r_tokens(lb):
    """Align mode ([ops] _commit_kda_state_kernel, ALIGN_MODE): the boundary
    slot receives the state after the first min(R, m) tokens, which is the
    verify's running state (S0 itself for R = 0) and the plain commit of that
    many tokens bit for bit; the final slot receives the committed state; the
    source slot keeps S0."""
    cfg = _tiny(B=4, slots=16, K=8, lower_bound=lb)
    prob = make_problem(cfg)
    meta = prob.meta
    B, H = cfg.B, cfg.H
    hl = host_layer(prob, 0)
    res = run_verify(prob, hl, want_running=True)
    lens = np.minimum(np.diff(meta.query_start_loc), cfg.Q)
    acc = np.minimum(np.maximum(meta.num_accepted, 0), lens)
    used = {int(x) for x in meta.state_indices if x > 0}
    free = [x for x in range(1, cfg.slots) if x not in used]
    final = np.array(free[:B], np.int32)
    bnd = np.array(free[B:2 * B], np.int32)
    R = np.array([0, 1, 2, 9], np.int32)  # none, inside the window, past it
    S0 = hl.state.copy()
    bexact = np.full((B, H, cfg.K, cfg.K), np.nan)
    exact = run_commit(prob, hl, want_exact=True, final_state_indices=final, boundary_state_indices=bnd,
                       boundary_recovery_lens=R, boundary_exact=bexact)
    # the plain commit of min(R, m) and of m tokens, on copies
    plain = {}
    for name, counts in (("boundary", np.minimum(R, acc)), ("final", acc)):
        hl2 = host_layer(prob, 0)
        hl2.corr[...] = hl.corr
        hl2.key_gate[...] = hl.key_gate
        hl2.state[...] = S0
        saved = meta.num_accepted
        meta.num_accepted = counts.astype(np.int32)
        run_commit(prob, hl2)
        meta.num_accepted = saved
        plain[name] = hl2.state
    checked = 0
    for b in range(B):
        s = int(meta.state_indices[b])
        if s <= 0 or acc[b] == 0:
            np.testing.assert_array_equal(hl.state[final[b]], S0[final[b]])
            np.testing.assert_array_equal(hl.state[bnd[b]], S0[bnd[b]])
            continue
        np.testing.assert_array_equal(hl.state[s], S0[s])  # the source keeps S0
        rb = min(int(R[b]), int(acc[b]))
        for h in range(H):
            np.testing.assert_array_equal(hl.state[bnd[b], h], plain["boundary"][s, h])
            np.testing.assert_array_equal(hl.state[final[b], h], plain["final"][s, h])
            np.testing.assert_array_equal(hl.state[final[b], h], exact[b, h].astype(np.float32))
            np.testing.assert_array_equal(hl.state[bnd[b], h], bexact[b, h].astype(np.float32))
            if rb == 0:
                np.testing.assert_array_equal(hl.state[bnd[b], h], S0[s, h])
            else:
                ref = res["running_state"][b, h, rb - 1]
                np.testing.assert_allclose(hl.state[bnd[b], h], ref, rtol=0, atol=2e-6 * np.abs(ref).max())
            checked += 1
    assert checked >= 4


def test_align_commit_null_final_slot_writes_nothing():
    prob = make_problem(_tiny(B=4, slots=16))
    meta = prob.meta
    meta.num_accepted[:] = np.minimum(np.diff(meta.query_start_loc), 4)
    hl = host_layer(prob, 0)
    run_verify(prob, hl)
    before = hl.state.copy()
    B = prob.cfg.B
    final = np.zeros(B, np.int32)  # every final slot null
    bnd = np.arange(10, 10 + B, dtype=np.int32)
    run_commit(prob, hl, final_state_indices=final, boundary_state_indices=bnd,
               boundary_recovery_lens=np.ones(B, np.int32))
    np.testing.assert_array_equal(hl.state, before)


def test_commit_zero_accepted_and_null_are_bit_identical():
    prob = make_problem(_tiny(B=4, slots=8))
    meta = prob.meta
    meta.num_accepted[:] = 0
    meta.num_accepted[1] = 2
    meta.state_indices[1] = -1  # null slot with accepted tokens: still nothing
    hl = host_layer(prob, 0)
    run_verify(prob, hl)
    before = hl.state.copy()
    run_commit(prob, hl)
    np.testing.assert_array_equal(hl.state, before)


def test_null_slot_writes_zero_outputs_only():
    prob = make_problem(_tiny(B=4, slots=8))
    meta = prob.meta
    meta.state_indices[2] = 0
    hl = host_layer(prob, 0)
    hl.out[...] = 0x7FA5
    hl.corr.view(np.uint32)[...] = 0x7FC0DEAD
    hl.key_gate[...] = 0x7FA5
    cs_before = hl.conv_state.copy()
    run_verify(prob, hl)
    bos, eos = int(meta.query_start_loc[2]), int(meta.query_start_loc[3])
    assert (hl.out[bos:eos] == 0).all()
    # row 0 (the null slot's row) of the records and slot 0's conv state untouched
    assert (hl.corr[0].view(np.uint32) == 0x7FC0DEAD).all()
    assert (hl.key_gate[0] == 0x7FA5).all()
    np.testing.assert_array_equal(hl.conv_state[0], cs_before[0])


def test_delta_rule_invariant_no_decay_full_beta():
    """g = 0 (A_log = -inf) and sigmoid(raw_beta) = 1: one step gives
    S_1 k^ - v = (S_0 k^ - v) * eps / (|k|^2 + eps), i.e. S_1 k^ = v up to eps."""
    cfg = _tiny(B=3, K=8, slots=6)
    prob = make_problem(cfg)
    prob.A_log.fill_(-math.inf)
    H, K = cfg.H, cfg.K
    prob.fused[0, :, 4 * H * K: 4 * H * K + H] = 40.0  # sigmoid(40) rounds to 1 in double
    hl = host_layer(prob, 0)
    res = run_verify(prob, hl, want_running=True, want_post_conv=True)
    meta = prob.meta
    for b in range(cfg.B):
        bos = int(meta.query_start_loc[b])
        s = int(meta.state_indices[b])
        for h in range(H):
            k = res["post_conv"][bos, H * K + h * K: H * K + (h + 1) * K]
            v = res["post_conv"][bos, 2 * H * K + h * K: 2 * H * K + (h + 1) * K]
            kk = float(k @ k)
            kh = k / math.sqrt(kk + 1e-6)
            S0 = hl.state[s, h].astype(np.float64)
            S1 = res["running_state"][b, h, 0]
            np.testing.assert_allclose(S1 @ kh - v, (S0 @ kh - v) * 1e-6 / (kk + 1e-6),
                                       rtol=1e-6, atol=1e-15)
            assert np.abs(S1 @ kh - v).max() < 1e-5


def test_output_closed_form_from_zero_state():
    """S_0 = 0, no decay, and q = k: o_1 = beta v k^.q^ = beta v |k|^2 / (|k|^2 + eps) / sqrt(K)."""
    cfg = _tiny(B=2, K=8, slots=4, conv_offsets=False)
    prob = make_problem(cfg)
    H, K = cfg.H, cfg.K
    prob.A_log.fill_(-math.inf)
    prob.state.zero_()
    # identical q and k channels: same weights, same inputs, same history
    cw = prob.conv_weight[0]
    cw[H * K: 2 * H * K] = cw[: H * K]
    f = prob.fused[0]
    f[:, H * K: 2 * H * K] = f[:, : H * K]
    cs = prob.conv_state[0]
    cs[:, H * K: 2 * H * K] = cs[:, : H * K]
    hl = host_layer(prob, 0)
    res = run_verify(prob, hl, want_exact=True, want_post_conv=True)
    meta = prob.meta
    for b in range(cfg.B):
        bos = int(meta.query_start_loc[b])
        for h in range(H):
            k = res["post_conv"][bos, H * K + h * K: H * K + (h + 1) * K]
            v = res["post_conv"][bos, 2 * H * K + h * K: 2 * H * K + (h + 1) * K]
            beta = expit(brute.bf16_values(hl.fused[bos, 4 * H * K + h]))
            kk = float(k @ k)
            ref = beta * v * kk / (kk + 1e-6) / math.sqrt(K)
            np.testing.assert_allclose(res["out_exact"][bos, h * K:(h + 1) * K], ref,
                                       rtol=1e-12, atol=1e-15)


# --------------------------------------------------------------------------- conv

@pytest.mark.parametrize("dim_first", [True, False])
def test_conv_unit_taps(dim_first):
    """w = e_{W-1}: the conv output is SiLU of the newest input; w = e_0: it is
    SiLU of the oldest tap of the window, i.e. the history read at offset a-1."""
    cfg = _tiny(B=3, K=8, slots=6, conv_dim_first=dim_first)
    for tap in (cfg.W - 1, 0):
        prob = make_problem(cfg)
        prob.conv_weight.zero_()
        prob.conv_weight[0, :, tap] = 1.0
        fresh = host_layer(prob, 0)
        hl = host_layer(prob, 0)
        res = run_verify(prob, hl, want_post_conv=True)
        meta = prob.meta
        for b in range(cfg.B):
            it = _item_inputs(prob, fresh, b, 0)
            seq = np.concatenate([it["hist"], it["x"]], axis=0)
            for t in range(it["n"]):
                src = seq[t + tap]
                brute.assert_codes_exact(_codes(res["post_conv"][it["bos"] + t, it["chans"]]), src)


@pytest.mark.parametrize("dim_first", [True, False])
def test_conv_state_roll_is_bit_copy(dim_first):
    cfg = _tiny(B=4, K=8, slots=8, conv_dim_first=dim_first)
    prob = make_problem(cfg)
    fresh = host_layer(prob, 0)
    hl = host_layer(prob, 0)
    run_verify(prob, hl)
    meta = prob.meta
    Lc, W = cfg.conv_len, cfg.W
    C = cfg.conv_dim
    for b in range(cfg.B):
        s = int(meta.state_indices[b])
        bos = int(meta.query_start_loc[b])
        n = min(int(meta.query_start_loc[b + 1]) - bos, cfg.Q)
        a = min(max(int(meta.num_accepted_prev[b]), 1), cfg.Q)
        old = fresh.conv_state[s] if dim_first else fresh.conv_state[s].T  # -> [C, Lc]
        new = hl.conv_state[s] if dim_first else hl.conv_state[s].T
        seq = np.concatenate([old[:, a - 1: a - 1 + W - 1], fresh.fused[bos: bos + n, :C].T], axis=1)
        np.testing.assert_array_equal(new[:, : W - 2 + n], seq[:, 1: W - 1 + n])
        np.testing.assert_array_equal(new[:, W - 2 + n:], old[:, W - 2 + n:])


def test_two_verifies_equal_one_over_the_joined_window():
    """Verify x_1..x_n1, accept all n1 (conv offset n1), verify x_n1+1..x_n: the
    second window's conv outputs equal those of one verify over x_1..x_n."""
    cfg = _tiny(B=2, K=8, slots=4, Q=4)
    n1, n2 = 2, 2
    prob = make_problem(cfg)
    H, K = cfg.H, cfg.K
    meta = prob.meta
    B = cfg.B
    # joined: each request has n1 + n2 tokens; rows 0..3 for b=0, 4..7 for b=1
    joined_qsl = np.arange(0, (n1 + n2) * (B + 1), n1 + n2, dtype=np.int32)
    T = int(joined_qsl[-1])
    assert prob.fused.shape[1] >= T or True
    g = torch.Generator().manual_seed(5)
    fused = (torch.randn((T, prob.fused.shape[2]), generator=g)).to(torch.bfloat16)
    from workloads import to_bits
    fb = to_bits(fused)

    def run(rows, qsl, prev, cs):
        hl = host_layer(prob, 0)
        hl.fused = np.ascontiguousarray(fb[rows])
        hl.out = np.zeros((len(rows), H * K), np.uint16)
        hl.conv_state = cs
        meta.query_start_loc = qsl
        meta.num_accepted_prev = prev
        res = run_verify(prob, hl, want_post_conv=True)
        return res["post_conv"], hl.conv_state

    cs0 = host_layer(prob, 0).conv_state.copy()
    ones = np.ones(B, np.int32)
    full, _ = run(np.arange(T), joined_qsl, ones, cs0.copy())
    first_rows = np.concatenate([np.arange(b * 4, b * 4 + n1) for b in range(B)])
    second_rows = np.concatenate([np.arange(b * 4 + n1, b * 4 + 4) for b in range(B)])
    qsl1 = np.arange(0, n1 * (B + 1), n1, dtype=np.int32)
    _, cs1 = run(first_rows, qsl1, ones, cs0.copy())
    second, _ = run(second_rows, np.arange(0, n2 * (B + 1), n2, dtype=np.int32),
                    np.full(B, n1, np.int32), cs1)
    for b in range(B):
        np.testing.assert_array_equal(second[b * n2:(b + 1) * n2], full[b * 4 + n1: b * 4 + 4])


def test_tokens_past_the_window_are_ignored():
    """A query longer than Q verifies only its first Q tokens; the rows past Q
    are not written."""
    cfg = _tiny(B=2, K=8, slots=4)
    prob = make_problem(cfg)
    meta = prob.meta
    Q = cfg.Q
    from workloads import to_bits
    g = torch.Generator().manual_seed(9)
    rows = 2 * Q + 2
    fb = to_bits(torch.randn((rows, prob.fused.shape[2]), generator=g).to(torch.bfloat16))
    H, K = cfg.H, cfg.K

    def run(qsl):
        hl = host_layer(prob, 0)
        hl.fused = fb
        hl.out = np.full((rows, H * K), 0x7FA5, np.uint16)
        meta.query_start_loc = np.array(qsl, np.int32)
        run_verify(prob, hl)
        return hl.out

    exact_q = run([0, Q, 2 * Q])              # request 0 has exactly Q tokens
    longer = run([0, Q + 2, 2 * Q + 2])       # request 0 has Q + 2 tokens
    np.testing.assert_array_equal(longer[:Q], exact_q[:Q])
    assert (longer[Q: Q + 2] == 0x7FA5).all()
    assert (longer[Q + 2:] != 0x7FA5).all()


def test_thread_count_does_not_change_results():
    prob = make_problem(CONFIGS["C0"])
    a = host_layer(prob, 0)
    b = host_layer(prob, 0)
    ra = run_verify(prob, a, want_exact=True, num_threads=1)
    rb = run_verify(prob, b, want_exact=True, num_threads=4)
    np.testing.assert_array_equal(ra["out_exact"], rb["out_exact"])
    np.testing.assert_array_equal(a.corr, b.corr)
    np.testing.assert_array_equal(a.key_gate, b.key_gate)
    np.testing.assert_array_equal(a.conv_state, b.conv_state)
