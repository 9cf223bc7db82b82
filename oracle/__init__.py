"""TEST INFRASTRUCTURE ONLY -- the double-precision CPU oracle.

A plain restatement, in C (``kda_oracle.c``), of the Kimi Delta Attention
RecoverSSM speculative verify and accepted-state commit from the vLLM pages
("vLLM/vllm/models/kimi_k3/nvidia/ops/recoverssm.py": ``_kda_gate``,
``_kda_recurrent_step``, ``_kda_recoverssm_verify_kernel``,
``_commit_kda_state_kernel``; "vllm.models.kimi_k3.nvidia.recoverssm.kernels":
``CuteRecoverSSMVerify.__call__`` for the fused short convolution).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA
library and never imports it.

Every function here takes numpy arrays: bf16 data as ``uint16`` bit patterns,
fp32 data as ``float32``, index data as ``int32``.  Pins: ``tests/test_oracle_pins.py``
(closed forms, special cases, invariants, an independent matrix-form brute
force at K=V=4).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FP contraction) and return the path."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_f64 = ctypes.c_double


class _VerifyArgs(ctypes.Structure):
    _fields_ = [
        ("B", _i32), ("H", _i32), ("K", _i32), ("V", _i32), ("Q", _i32), ("W", _i32),
        ("T", _i32), ("null_block_id", _i32),
        ("num_slots", _i64), ("num_record_rows", _i64),
        ("mixed_qkv", _p), ("qkv_row_stride", _i64),
        ("raw_gate", _p), ("gate_row_stride", _i64),
        ("raw_beta", _p), ("beta_row_stride", _i64),
        ("A_log", _p), ("dt_bias", _p),
        ("use_lower_bound", _i32), ("lower_bound", _f64),
        ("conv_weight", _p), ("conv_weight_is_fp32", _i32),
        ("conv_state", _p), ("conv_dim_first", _i32), ("conv_slot_stride", _i64),
        ("state", _p), ("state_slot_stride", _i64),
        ("query_start_loc", _p), ("state_indices", _p), ("record_indices", _p),
        ("num_accepted_prev", _p), ("item_mask", _p),
        ("out", _p), ("out_row_stride", _i64), ("out_exact", _p),
        ("corr", _p), ("corr_row_stride", _i64), ("corr_exact", _p),
        ("key_gate", _p), ("kg_row_stride", _i64),
        ("running_state", _p), ("post_conv", _p),
        ("num_threads", _i32),
    ]


class _CommitArgs(ctypes.Structure):
    _fields_ = [
        ("B", _i32), ("H", _i32), ("K", _i32), ("V", _i32), ("Q", _i32), ("null_block_id", _i32),
        ("num_slots", _i64), ("num_record_rows", _i64),
        ("state", _p), ("state_slot_stride", _i64), ("state_exact", _p),
        ("corr", _p), ("corr_row_stride", _i64),
        ("key_gate", _p), ("kg_row_stride", _i64),
        ("A_log", _p), ("dt_bias", _p),
        ("use_lower_bound", _i32), ("lower_bound", _f64),
        ("query_start_loc", _p), ("state_indices", _p), ("record_indices", _p),
        ("num_accepted", _p), ("item_mask", _p),
        ("num_threads", _i32),
        ("final_state_indices", _p), ("boundary_state_indices", _p), ("boundary_recovery_lens", _p),
        ("boundary_exact", _p),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.kda_oracle_verify.argtypes = [ctypes.POINTER(_VerifyArgs)]
            lib.kda_oracle_verify.restype = ctypes.c_int
            lib.kda_oracle_commit.argtypes = [ctypes.POINTER(_CommitArgs)]
            lib.kda_oracle_commit.restype = ctypes.c_int
            lib.kda_oracle_bf16_round.argtypes = [ctypes.c_double]
            lib.kda_oracle_bf16_round.restype = ctypes.c_uint16
            lib.kda_oracle_gate.argtypes = [ctypes.c_double] * 3 + [ctypes.c_int, ctypes.c_double]
            lib.kda_oracle_gate.restype = ctypes.c_double
            lib.kda_oracle_conv_silu_bf16.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64, ctypes.c_int]
            lib.kda_oracle_conv_silu_bf16.restype = None
            _lib = lib
    return _lib


def _ptr(a, dtype=None):
    if a is None:
        return None
    if dtype is not None and a.dtype != dtype:
        raise TypeError(f"oracle: expected {dtype}, got {a.dtype}")
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("oracle: arrays must be C-contiguous (row strides are passed explicitly)")
    return a.ctypes.data


def _row_stride(a):
    return a.strides[0] // a.itemsize


def bf16_round(x: float) -> int:
    """bf16 bits of ``x`` rounded to nearest even (straight from double)."""
    return int(_load().kda_oracle_bf16_round(float(x)))


def gate(raw_g: float, dt_bias: float, A: float, lower_bound: float | None = None) -> float:
    """The KDA gate g (``_kda_gate``) in double."""
    use_lb = lower_bound is not None
    return float(_load().kda_oracle_gate(raw_g, dt_bias, A, int(use_lb), float(lower_bound or 0.0)))


def conv_silu_bf16(w, x) -> np.ndarray:
    """bf16 codes of SiLU(sum_j w_j x_j) by the plain definition in double,
    rounded once; w, x: [n, W] taps oldest first (values, any float dtype)."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    x = np.ascontiguousarray(x, dtype=np.float64)
    if w.shape != x.shape or w.ndim != 2:
        raise ValueError("oracle: w and x must both be [n, W]")
    out = np.empty(w.shape[0], np.uint16)
    _load().kda_oracle_conv_silu_bf16(w.ctypes.data, x.ctypes.data, out.ctypes.data, w.shape[0], w.shape[1])
    return out


def verify(*, H, K, Q, W, mixed_qkv, raw_gate, raw_beta, A_log, dt_bias, lower_bound,
           conv_weight, conv_state, conv_dim_first, state, corr, key_gate, out,
           query_start_loc, state_indices, record_indices=None, num_accepted_prev=None,
           null_block_id=0, item_mask=None, want_exact=False, want_running=False,
           want_post_conv=False, num_threads=0):
    """One layer's verify.  ``mixed_qkv`` [T, >=3HK], ``raw_gate`` [T, >=HK],
    ``raw_beta`` [T, >=H] may be column windows of one buffer (pass them as
    2-D arrays whose row stride is the buffer's; the first column is element 0).

    Writes ``out`` (bf16 bits), ``corr`` (fp32), ``key_gate`` (bf16 bits) and
    ``conv_state`` (bf16 bits) in place; ``state`` is read only.  Returns a
    dict with the optional exact (double) outputs."""
    lib = _load()
    B = int(state_indices.shape[0])
    T = int(out.shape[0])
    V = K
    res = {}
    out_exact = np.zeros((T, H * V), np.float64) if want_exact else None
    corr_exact = np.full(corr.shape, np.nan, np.float64) if want_exact else None
    running = np.zeros((B, H, Q, V, K), np.float64) if want_running else None
    post = np.full((T, 3 * H * K), np.nan, np.float64) if want_post_conv else None
    a = _VerifyArgs()
    a.B, a.H, a.K, a.V, a.Q, a.W, a.T = B, H, K, V, Q, W, T
    a.null_block_id = null_block_id
    a.num_slots = state.shape[0]
    a.num_record_rows = corr.shape[0]
    for name, arr, dt in (("mixed_qkv", mixed_qkv, np.uint16), ("raw_gate", raw_gate, np.uint16),
                          ("raw_beta", raw_beta, np.uint16)):
        if arr.dtype != dt or arr.strides[1] != arr.itemsize:
            raise ValueError(f"oracle: {name} must be uint16 with unit column stride")
        setattr(a, name, arr.ctypes.data)
    a.qkv_row_stride = _row_stride(mixed_qkv)
    a.gate_row_stride = _row_stride(raw_gate)
    a.beta_row_stride = _row_stride(raw_beta)
    a.A_log = _ptr(A_log, np.float32)
    a.dt_bias = _ptr(dt_bias, np.float32)
    a.use_lower_bound = int(lower_bound is not None)
    a.lower_bound = float(lower_bound or 0.0)
    a.conv_weight = _ptr(conv_weight)
    a.conv_weight_is_fp32 = int(conv_weight.dtype == np.float32)
    a.conv_state = _ptr(conv_state, np.uint16)
    a.conv_dim_first = int(conv_dim_first)
    a.conv_slot_stride = _row_stride(conv_state)
    a.state = _ptr(state, np.float32)
    a.state_slot_stride = _row_stride(state)
    a.query_start_loc = _ptr(query_start_loc, np.int32)
    a.state_indices = _ptr(state_indices, np.int32)
    a.record_indices = _ptr(record_indices, np.int32)
    a.num_accepted_prev = _ptr(num_accepted_prev, np.int32)
    a.item_mask = _ptr(item_mask, np.uint8)
    a.out = _ptr(out, np.uint16)
    a.out_row_stride = _row_stride(out)
    a.out_exact = _ptr(out_exact)
    a.corr = _ptr(corr, np.float32)
    a.corr_row_stride = _row_stride(corr)
    a.corr_exact = _ptr(corr_exact)
    a.key_gate = _ptr(key_gate, np.uint16)
    a.kg_row_stride = _row_stride(key_gate)
    a.running_state = _ptr(running)
    a.post_conv = _ptr(post)
    a.num_threads = num_threads
    st = lib.kda_oracle_verify(ctypes.byref(a))
    if st != 0:
        raise RuntimeError(f"oracle verify: status {st}")
    res["out_exact"], res["corr_exact"], res["running_state"], res["post_conv"] = (
        out_exact, corr_exact, running, post)
    return res


def commit(*, H, K, Q, state, corr, key_gate, A_log, dt_bias, lower_bound,
           query_start_loc, state_indices, num_accepted, record_indices=None,
           null_block_id=0, item_mask=None, want_exact=False, num_threads=0,
           final_state_indices=None, boundary_state_indices=None, boundary_recovery_lens=None,
           boundary_exact=None):
    """One layer's commit: folds each request's first
    min(max(num_accepted, 0), query_len) records into ``state`` (fp32, in
    place).  Returns the unrounded double states [B, H, V, K] when asked.

    Align mode: the committed state goes to ``final_state_indices[b]`` (None:
    the source slot), and a live ``boundary_state_indices[b]`` receives the
    state after the first ``boundary_recovery_lens[b]`` tokens (its unrounded
    value into ``boundary_exact`` [B, H, V, K] float64 when given)."""
    lib = _load()
    B = int(state_indices.shape[0])
    V = K
    exact = np.full((B, H, V, K), np.nan, np.float64) if want_exact else None
    a = _CommitArgs()
    a.B, a.H, a.K, a.V, a.Q = B, H, K, V, Q
    a.null_block_id = null_block_id
    a.num_slots = state.shape[0]
    a.num_record_rows = corr.shape[0]
    a.state = _ptr(state, np.float32)
    a.state_slot_stride = _row_stride(state)
    a.state_exact = _ptr(exact)
    a.corr = _ptr(corr, np.float32)
    a.corr_row_stride = _row_stride(corr)
    a.key_gate = _ptr(key_gate, np.uint16)
    a.kg_row_stride = _row_stride(key_gate)
    a.A_log = _ptr(A_log, np.float32)
    a.dt_bias = _ptr(dt_bias, np.float32)
    a.use_lower_bound = int(lower_bound is not None)
    a.lower_bound = float(lower_bound or 0.0)
    a.query_start_loc = _ptr(query_start_loc, np.int32)
    a.state_indices = _ptr(state_indices, np.int32)
    a.record_indices = _ptr(record_indices, np.int32)
    a.num_accepted = _ptr(num_accepted, np.int32)
    a.item_mask = _ptr(item_mask, np.uint8)
    a.num_threads = num_threads
    a.final_state_indices = _ptr(final_state_indices, np.int32)
    a.boundary_state_indices = _ptr(boundary_state_indices, np.int32)
    a.boundary_recovery_lens = _ptr(boundary_recovery_lens, np.int32)
    if boundary_exact is not None:
        if boundary_exact.dtype != np.float64 or boundary_exact.shape != (B, H, V, K):
            raise ValueError("boundary_exact must be float64 [B, H, V, K]")
    a.boundary_exact = _ptr(boundary_exact)
    st = lib.kda_oracle_commit(ctypes.byref(a))
    if st != 0:
        raise RuntimeError(f"oracle commit: status {st}")
    return exact
