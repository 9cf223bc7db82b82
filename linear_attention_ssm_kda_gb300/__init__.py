"""KDA RecoverSSM speculative verify and accepted-state commit on GB300.

A thin ctypes binding over ``libkda.so`` (C ABI in ``include/kda.h``): it
reads shapes, strides, dtypes and device pointers off torch tensors and
forwards them; every step of the computation runs in the library's sm_103a
kernels.  PyTorch only owns the memory and the stream.  There is no CPU path:
if the library is not built, importing the functions raises.

Operations follow the vLLM Kimi-K3 RecoverSSM pages:
``verify`` is "vllm.models.kimi_k3.nvidia.recoverssm.kernels",
``CuteRecoverSSMVerify.__call__`` (short conv fused in front of
"vLLM/vllm/models/kimi_k3/nvidia/ops/recoverssm.py", ``kda_recoverssm_verify``);
``CommitContext`` is that ops page's ``KDARecoverSSMCommitContext``
(``create`` / ``commit``), folding all layers in one launch.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Sequence

import torch

__all__ = [
    "commit_noalloc",
    "KdaError", "lib_path", "load_library", "verify", "CommitContext", "workspace_bytes",
    "new_workspace", "read_device_error", "last_error", "verify_scratch_bytes", "new_verify_scratch",
    "DEVERR_SLOT_RANGE", "DEVERR_ROW_RANGE", "DEVERR_TOKEN_RANGE", "DEVERR_TIMEOUT", "DEVERR_MISALIGNED",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_MISALIGNED, KDA_ERR_CUDA, KDA_ERR_DEVICE = range(6)
GATE_SOFTPLUS, GATE_LOWER_BOUND = 0, 1
CONV_DIM_FIRST, CONV_SEQ_FIRST = 0, 1
DTYPE_BF16, DTYPE_FP32 = 0, 1
DEVERR_SLOT_RANGE, DEVERR_ROW_RANGE, DEVERR_TOKEN_RANGE, DEVERR_TIMEOUT, DEVERR_MISALIGNED = 1, 2, 4, 8, 16
_STATUS = {1: "invalid argument", 2: "unsupported", 3: "misaligned", 4: "CUDA error", 5: "device error"}


class KdaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libkda: {_STATUS.get(status, status)}: {message}")
        self.status = status


_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


class VerifyArgs(ctypes.Structure):
    """Mirror of ``kda_verify_args``."""
    _fields_ = [
        ("B", _i32), ("H", _i32), ("K", _i32), ("V", _i32), ("Q", _i32), ("W", _i32), ("T", _i32),
        ("null_block_id", _i32), ("num_slots", _i64), ("num_record_rows", _i64),
        ("mixed_qkv", _p), ("qkv_row_stride", _i64),
        ("raw_gate", _p), ("gate_row_stride", _i64),
        ("raw_beta", _p), ("beta_row_stride", _i64),
        ("out", _p), ("out_row_stride", _i64),
        ("A_log", _p), ("dt_bias", _p), ("gate_mode", _i32), ("lower_bound", ctypes.c_float),
        ("conv_weight", _p), ("conv_weight_dtype", _i32),
        ("conv_state", _p), ("conv_layout", _i32), ("conv_slot_stride", _i64),
        ("state", _p), ("state_slot_stride", _i64),
        ("corr", _p), ("corr_row_stride", _i64),
        ("key_gate", _p), ("kg_row_stride", _i64),
        ("query_start_loc", _p), ("state_indices", _p), ("record_indices", _p),
        ("num_accepted_prev", _p), ("workspace", _p),
        ("scratch", _p), ("scratch_bytes", _i64), ("variant", _i32),
    ]


VARIANTS = {"auto": 0, "cuda_core": 1, "tcgen05": 2}


class DebugArgs(ctypes.Structure):
    """Mirror of ``kda_debug_args``."""
    _fields_ = [("wait_limit_ns", _i64), ("withhold_item", _i32), ("cta_times", _p)]


class AlignArgs(ctypes.Structure):
    """Mirror of ``kda_align_args``."""
    _fields_ = [("final_state_indices", _p), ("boundary_state_indices", _p), ("boundary_recovery_lens", _p)]


class FoldArgs(ctypes.Structure):
    """Mirror of ``kda_fold_args``."""
    _fields_ = [("query_start_loc", _p), ("num_accepted", _p), ("record_indices", _p)]


class CommitArgs(ctypes.Structure):
    """Mirror of ``kda_commit_args``."""
    _fields_ = [
        ("L", _i32), ("B", _i32), ("H", _i32), ("K", _i32), ("V", _i32), ("Q", _i32),
        ("null_block_id", _i32), ("num_slots", _i64), ("num_record_rows", _i64),
        ("state_base", _p), ("state_slot_stride", _p), ("corr_base", _p), ("corr_row_stride", _p),
        ("kg_base", _p), ("kg_row_stride", _p), ("A_log", _p), ("dt_bias", _p),
        ("gate_mode", _i32), ("lower_bound", ctypes.c_float),
        ("query_start_loc", _p), ("state_indices", _p), ("record_indices", _p),
        ("num_accepted", _p), ("workspace", _p),
    ]


_lib = None
_lib_lock = threading.Lock()


def lib_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libkda.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise ImportError(
                    f"libkda.so is not built ({_LIB_PATH}); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            lib = ctypes.CDLL(_LIB_PATH)
            lib.kda_verify.argtypes = [ctypes.POINTER(VerifyArgs), _p]
            lib.kda_verify.restype = ctypes.c_int
            lib.kda_verify_fold.argtypes = [ctypes.POINTER(VerifyArgs), ctypes.POINTER(FoldArgs), _p]
            lib.kda_verify_fold.restype = ctypes.c_int
            lib.kda_verify_debug.argtypes = [ctypes.POINTER(VerifyArgs), ctypes.POINTER(DebugArgs), _p]
            lib.kda_verify_debug.restype = ctypes.c_int
            lib.kda_commit.argtypes = [ctypes.POINTER(CommitArgs), _p]
            lib.kda_commit.restype = ctypes.c_int
            lib.kda_commit_align.argtypes = [ctypes.POINTER(CommitArgs), ctypes.POINTER(AlignArgs), _p]
            lib.kda_commit_align.restype = ctypes.c_int
            lib.kda_commit_noalloc.argtypes = [ctypes.POINTER(CommitArgs), _p]
            lib.kda_commit_noalloc.restype = ctypes.c_int
            lib.kda_workspace_bytes.argtypes = []
            lib.kda_workspace_bytes.restype = ctypes.c_size_t
            lib.kda_verify_scratch_bytes.argtypes = [_i32, _i32, _i32, _i32]
            lib.kda_verify_scratch_bytes.restype = ctypes.c_size_t
            lib.kda_read_device_error.argtypes = [_p, _p, ctypes.POINTER(_i32)]
            lib.kda_read_device_error.restype = ctypes.c_int
            lib.kda_last_error.argtypes = []
            lib.kda_last_error.restype = ctypes.c_char_p
            lib.kda_abi_version.argtypes = []
            lib.kda_abi_version.restype = _i32
            _lib = lib
    return _lib


def last_error() -> str:
    return load_library().kda_last_error().decode()


def _check(status: int) -> None:
    if status != KDA_OK:
        raise KdaError(status, last_error())


def workspace_bytes() -> int:
    return int(load_library().kda_workspace_bytes())


def verify_scratch_bytes(B: int, H: int, K: int, window: int) -> int:
    """Bytes of device scratch one verify call needs (the conv pass's output)."""
    return int(load_library().kda_verify_scratch_bytes(B, H, K, window))


def new_verify_scratch(B: int, H: int, K: int, window: int, device) -> torch.Tensor:
    """Device scratch for ``verify`` (allocated by torch on the current stream)."""
    return torch.empty(max(verify_scratch_bytes(B, H, K, window), 16), dtype=torch.uint8, device=device)


def new_workspace(device) -> torch.Tensor:
    """A zeroed device workspace: the error report and the verify's ticket
    counter (allocated by torch on the current stream)."""
    return torch.zeros((workspace_bytes() + 3) // 4, dtype=torch.int32, device=device)


def _stream_handle(device, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def read_device_error(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream and return the device error bits (0: none)."""
    flags = _i32(0)
    st = load_library().kda_read_device_error(
        ctypes.c_void_p(workspace.data_ptr()), ctypes.c_void_p(_stream_handle(workspace.device, stream)),
        ctypes.byref(flags))
    if st not in (KDA_OK, KDA_ERR_DEVICE):
        _check(st)
    return int(flags.value)


def _need(t: torch.Tensor, name: str, dtype, device, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if ndim is not None and t.ndim != ndim:
        raise ValueError(f"{name} must be {ndim}-D, got shape {tuple(t.shape)}")


def _inner_contiguous(t: torch.Tensor, name: str, dims: int) -> None:
    """The last ``dims`` dimensions must be densely packed row-major."""
    expect = 1
    for d in range(t.ndim - 1, t.ndim - 1 - dims, -1):
        if t.shape[d] > 1 and t.stride(d) != expect:
            raise ValueError(f"{name}: inner dimensions must be contiguous (strides {t.stride()})")
        expect *= t.shape[d]


def _ptr(t):
    return None if t is None else t.data_ptr()


def verify(*, mixed_qkv, raw_gate, raw_beta, A_log, dt_bias, lower_bound, state, correction,
           key_gate, query_start_loc, state_indices, conv_state, conv_weight, out, window,
           num_accepted_tokens=None, record_indices=None, conv_dim_first=True, null_block_id=0,
           workspace=None, stream=None, fold_query_start_loc=None, fold_num_accepted=None,
           fold_record_indices=None, scratch=None, variant: str = "auto", debug=None) -> None:
    """Verify ``state_indices.shape[0]`` requests of one KDA layer.

    ``mixed_qkv`` [T, 3HK] is the raw projection (before the convolution),
    ``raw_gate`` [T, HK], ``raw_beta`` [T, H], ``out`` [T, HV], all bf16 with
    unit column stride (rows may be views into a wider buffer, at any
    offset).  ``state`` fp32 [slots, H, V, K] (read only), ``correction`` fp32
    [rows, H, window, V], ``key_gate`` bf16 [rows, H, window, 2K],
    ``conv_state`` bf16 [slots, 3HK, window+2] (dim first) or
    [slots, window+2, 3HK], ``conv_weight`` bf16 or fp32 [3HK, 4].
    ``lower_bound`` None selects the softplus gate, a float the bounded one.
    Asynchronous on ``stream`` (default: the current stream).

    With ``fold_query_start_loc`` and ``fold_num_accepted`` (the previous
    step's query_start_loc [B+1] and accepted counts [B], and optionally its
    record rows ``fold_record_indices``) this is ``kda_verify_fold``: each
    request's pending records are first folded into its checkpoint, which is
    written back, and the verify runs on the folded state (on the CUDA cores).

    ``scratch`` is a device buffer of at least ``verify_scratch_bytes(B, H,
    K, window)`` bytes for the conv pass's output; when None, one is taken
    from torch's allocator on the launch stream for this call.  ``variant``
    ("auto", "cuda_core" or "tcgen05") picks the kernel of the products (the
    tensor cores need K = 128).  ``workspace`` (``new_workspace``) holds the
    device error report and the ticket counter that deals the items to the
    kernel's CTAs; when None, a fresh one is allocated for this call.  Calls
    that may overlap on different streams need different workspaces.

    ``debug`` = (withhold_item, wait_limit_ns[, cta_times]) calls
    ``kda_verify_debug`` instead (no fold): item ``withhold_item`` (-1: none)
    has its inputs withheld and every device wait gives up after
    wait_limit_ns (a test of the bounded waits, on the CUDA cores); an int64
    ``cta_times`` [>= 2 B H] receives each verify CTA's start and finish on
    the GPU's global timer (ns)."""
    dev = state.device
    if dev.type != "cuda":
        raise ValueError("verify runs on a CUDA device; state is on " + str(dev))
    _need(state, "state", torch.float32, dev, 4)
    slots, H, V, K = state.shape
    _inner_contiguous(state, "state", 3)
    _need(mixed_qkv, "mixed_qkv", torch.bfloat16, dev, 2)
    _need(raw_gate, "raw_gate", torch.bfloat16, dev, 2)
    _need(raw_beta, "raw_beta", torch.bfloat16, dev, 2)
    _need(out, "out", torch.bfloat16, dev, 2)
    T = mixed_qkv.shape[0]
    for name, t, width in (("mixed_qkv", mixed_qkv, 3 * H * K), ("raw_gate", raw_gate, H * K),
                           ("raw_beta", raw_beta, H), ("out", out, H * V)):
        if t.shape != (T, width):
            raise ValueError(f"{name} must have shape {(T, width)}, got {tuple(t.shape)}")
        if width > 1 and t.stride(1) != 1:
            raise ValueError(f"{name} must have unit column stride")
    _need(A_log, "A_log", torch.float32, dev)
    _need(dt_bias, "dt_bias", torch.float32, dev)
    if A_log.numel() != H or dt_bias.numel() != H * K or not A_log.is_contiguous() or not dt_bias.is_contiguous():
        raise ValueError("A_log must be contiguous [H] and dt_bias contiguous [H*K]")
    _need(correction, "correction", torch.float32, dev, 4)
    _need(key_gate, "key_gate", torch.bfloat16, dev, 4)
    rows = correction.shape[0]
    if correction.shape != (rows, H, window, V) or key_gate.shape != (rows, H, window, 2 * K):
        raise ValueError(f"records must be [rows, {H}, {window}, {V}] and [rows, {H}, {window}, {2 * K}]")
    _inner_contiguous(correction, "correction", 3)
    _inner_contiguous(key_gate, "key_gate", 3)
    _need(conv_state, "conv_state", torch.bfloat16, dev, 3)
    conv_len = window + 2
    cs_shape = (slots, 3 * H * K, conv_len) if conv_dim_first else (slots, conv_len, 3 * H * K)
    if tuple(conv_state.shape) != cs_shape:
        raise ValueError(f"conv_state must have shape {cs_shape}, got {tuple(conv_state.shape)}")
    _inner_contiguous(conv_state, "conv_state", 2)
    if conv_weight.dtype not in (torch.bfloat16, torch.float32) or conv_weight.device != dev:
        raise TypeError("conv_weight must be a bf16 or fp32 tensor on the state's device")
    if tuple(conv_weight.shape) != (3 * H * K, 4) or not conv_weight.is_contiguous():
        raise ValueError(f"conv_weight must be contiguous [{3 * H * K}, 4]")
    B = state_indices.shape[0]
    _need(query_start_loc, "query_start_loc", torch.int32, dev, 1)
    _need(state_indices, "state_indices", torch.int32, dev, 1)
    if query_start_loc.shape[0] != B + 1 or not query_start_loc.is_contiguous() or not state_indices.is_contiguous():
        raise ValueError("query_start_loc must be contiguous [B+1] and state_indices contiguous [B]")
    for name, t in (("record_indices", record_indices), ("num_accepted_tokens", num_accepted_tokens)):
        if t is not None:
            _need(t, name, torch.int32, dev, 1)
            if t.shape[0] < B or not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous with at least B entries")
    if workspace is not None:
        _need(workspace, "workspace", torch.int32, dev)
        if workspace.numel() * 4 < workspace_bytes() or not workspace.is_contiguous():
            raise ValueError("workspace must be contiguous with at least workspace_bytes() bytes")
    else:
        # the verify's ticket counter needs one; tied to the launch stream
        with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream(dev)):
            workspace = new_workspace(dev)
    fold = None
    if fold_query_start_loc is not None:
        if fold_num_accepted is None:
            raise ValueError("fold_num_accepted is required with fold_query_start_loc")
        _need(fold_query_start_loc, "fold_query_start_loc", torch.int32, dev, 1)
        if fold_query_start_loc.shape[0] != B + 1 or not fold_query_start_loc.is_contiguous():
            raise ValueError("fold_query_start_loc must be contiguous [B+1]")
        for name, t in (("fold_num_accepted", fold_num_accepted), ("fold_record_indices", fold_record_indices)):
            if t is not None:
                _need(t, name, torch.int32, dev, 1)
                if t.shape[0] < B or not t.is_contiguous():
                    raise ValueError(f"{name} must be contiguous with at least B entries")
        fold = FoldArgs()
        fold.query_start_loc = fold_query_start_loc.data_ptr()
        fold.num_accepted = fold_num_accepted.data_ptr()
        fold.record_indices = _ptr(fold_record_indices)

    a = VerifyArgs()
    a.B, a.H, a.K, a.V, a.Q, a.W, a.T = B, H, K, V, window, 4, T
    a.null_block_id = null_block_id
    a.num_slots, a.num_record_rows = slots, rows
    a.mixed_qkv, a.qkv_row_stride = mixed_qkv.data_ptr(), mixed_qkv.stride(0)
    a.raw_gate, a.gate_row_stride = raw_gate.data_ptr(), raw_gate.stride(0)
    a.raw_beta, a.beta_row_stride = raw_beta.data_ptr(), raw_beta.stride(0)
    a.out, a.out_row_stride = out.data_ptr(), out.stride(0)
    a.A_log, a.dt_bias = A_log.data_ptr(), dt_bias.data_ptr()
    a.gate_mode = GATE_SOFTPLUS if lower_bound is None else GATE_LOWER_BOUND
    a.lower_bound = 0.0 if lower_bound is None else float(lower_bound)
    a.conv_weight = conv_weight.data_ptr()
    a.conv_weight_dtype = DTYPE_FP32 if conv_weight.dtype == torch.float32 else DTYPE_BF16
    a.conv_state, a.conv_slot_stride = conv_state.data_ptr(), conv_state.stride(0)
    a.conv_layout = CONV_DIM_FIRST if conv_dim_first else CONV_SEQ_FIRST
    a.state, a.state_slot_stride = state.data_ptr(), state.stride(0)
    a.corr, a.corr_row_stride = correction.data_ptr(), correction.stride(0)
    a.key_gate, a.kg_row_stride = key_gate.data_ptr(), key_gate.stride(0)
    a.query_start_loc, a.state_indices = query_start_loc.data_ptr(), state_indices.data_ptr()
    a.record_indices, a.num_accepted_prev = _ptr(record_indices), _ptr(num_accepted_tokens)
    a.workspace = _ptr(workspace)
    if variant not in VARIANTS:
        raise ValueError(f"variant must be one of {sorted(VARIANTS)}")
    a.variant = VARIANTS[variant]
    need = verify_scratch_bytes(B, H, K, window)
    if scratch is None and T > 0:
        # tied to the launch stream, so torch reuses it only after this call's kernels
        with torch.cuda.stream(stream if stream is not None else torch.cuda.current_stream(dev)):
            scratch = torch.empty(need, dtype=torch.uint8, device=dev)
    if scratch is not None:
        if scratch.device != dev or not scratch.is_contiguous():
            raise ValueError("scratch must be a contiguous tensor on the state's device")
        a.scratch, a.scratch_bytes = scratch.data_ptr(), scratch.numel() * scratch.element_size()
    handle = ctypes.c_void_p(_stream_handle(dev, stream))
    if debug is not None:
        if fold is not None:
            raise ValueError("debug runs the plain verify (no fold)")
        d = DebugArgs()
        d.withhold_item, d.wait_limit_ns = int(debug[0]), int(debug[1])
        if len(debug) > 2 and debug[2] is not None:
            times = debug[2]
            if times.device != dev or times.dtype != torch.int64 or not times.is_contiguous() \
                    or times.numel() < 2 * B * H:
                raise ValueError("cta_times must be a contiguous int64 tensor of >= 2*B*H on the state's device")
            d.cta_times = times.data_ptr()
        _check(load_library().kda_verify_debug(ctypes.byref(a), ctypes.byref(d), handle))
    elif fold is None:
        _check(load_library().kda_verify(ctypes.byref(a), handle))
    else:
        _check(load_library().kda_verify_fold(ctypes.byref(a), ctypes.byref(fold), handle))


class CommitContext:
    """All KDA layers' states and verify records, for one-launch commits.

    ``states[l]`` fp32 [slots, H, V, K], ``corrections[l]`` fp32
    [rows, H, window, V], ``key_gates[l]`` bf16 [rows, H, window, 2K] (each
    layer may live anywhere; inner layouts must match), ``A_log`` fp32 [L, H],
    ``dt_bias`` fp32 [L, H*K] (or [L, H, K]).  The per-layer base addresses and
    strides go to the device once, here."""

    def __init__(self, states: Sequence[torch.Tensor], corrections: Sequence[torch.Tensor],
                 key_gates: Sequence[torch.Tensor], A_log: torch.Tensor, dt_bias: torch.Tensor,
                 lower_bound: float | None, window: int):
        if not states:
            raise ValueError("KDA commit requires at least one layer")
        if not (len(states) == len(corrections) == len(key_gates)):
            raise ValueError("states, corrections and key_gates need one entry per layer")
        ref = states[0]
        dev = ref.device
        L = len(states)
        slots, H, V, K = ref.shape
        rows = corrections[0].shape[0]
        for l in range(L):
            _need(states[l], f"states[{l}]", torch.float32, dev, 4)
            _need(corrections[l], f"corrections[{l}]", torch.float32, dev, 4)
            _need(key_gates[l], f"key_gates[{l}]", torch.bfloat16, dev, 4)
            if states[l].shape != ref.shape:
                raise ValueError("layers need matching state shapes")
            if corrections[l].shape != (rows, H, window, V) or key_gates[l].shape != (rows, H, window, 2 * K):
                raise ValueError("layers need matching record shapes")
            _inner_contiguous(states[l], f"states[{l}]", 3)
            _inner_contiguous(corrections[l], f"corrections[{l}]", 3)
            _inner_contiguous(key_gates[l], f"key_gates[{l}]", 3)
        _need(A_log, "A_log", torch.float32, dev)
        _need(dt_bias, "dt_bias", torch.float32, dev)
        if A_log.numel() != L * H or dt_bias.numel() != L * H * K:
            raise ValueError("A_log must be [L, H] and dt_bias [L, H*K]")
        self.states, self.corrections, self.key_gates = tuple(states), tuple(corrections), tuple(key_gates)
        self.A_log = A_log.contiguous()
        self.dt_bias = dt_bias.contiguous()
        self.lower_bound = lower_bound
        self.window = window
        self.L, self.H, self.K, self.V, self.slots, self.rows = L, H, K, V, slots, rows
        self.device = dev

        def table(vals):
            return torch.tensor(vals, dtype=torch.int64, device=dev)

        self.state_base = table([t.data_ptr() for t in states])
        self.state_stride = table([t.stride(0) for t in states])
        self.corr_base = table([t.data_ptr() for t in corrections])
        self.corr_stride = table([t.stride(0) for t in corrections])
        self.kg_base = table([t.data_ptr() for t in key_gates])
        self.kg_stride = table([t.stride(0) for t in key_gates])

    def commit(self, num_accepted_tokens: torch.Tensor, state_indices: torch.Tensor,
               query_start_loc: torch.Tensor, record_indices: torch.Tensor | None = None,
               null_block_id: int = 0, workspace: torch.Tensor | None = None, stream=None,
               final_state_indices: torch.Tensor | None = None,
               boundary_state_indices: torch.Tensor | None = None,
               boundary_recovery_lens: torch.Tensor | None = None) -> None:
        """Fold each request's first min(max(accepted, 0), query_len) records
        into every layer's state (one kernel launch, asynchronous).

        Align mode (``kda_commit_align``): the committed state goes to
        ``final_state_indices[b]`` (default the source slot; a null one writes
        nothing) and a live ``boundary_state_indices[b]`` receives the state
        after the first ``boundary_recovery_lens[b]`` tokens."""
        dev = self.device
        B = state_indices.shape[0]
        _need(num_accepted_tokens, "num_accepted_tokens", torch.int32, dev, 1)
        _need(state_indices, "state_indices", torch.int32, dev, 1)
        _need(query_start_loc, "query_start_loc", torch.int32, dev, 1)
        if query_start_loc.shape[0] != B + 1 or num_accepted_tokens.shape[0] < B:
            raise ValueError("commit metadata is incompatible: query_start_loc [B+1], num_accepted [B]")
        for t in (num_accepted_tokens, state_indices, query_start_loc):
            if not t.is_contiguous():
                raise ValueError("commit metadata must be contiguous")
        if record_indices is not None:
            _need(record_indices, "record_indices", torch.int32, dev, 1)
            if record_indices.shape[0] < B or not record_indices.is_contiguous():
                raise ValueError("record_indices is too short")
        if workspace is not None:
            _need(workspace, "workspace", torch.int32, dev)
        align = None
        if final_state_indices is not None or boundary_state_indices is not None:
            if boundary_state_indices is not None and boundary_recovery_lens is None:
                raise ValueError("boundary_recovery_lens is required with boundary_state_indices")
            for name, t in (("final_state_indices", final_state_indices),
                            ("boundary_state_indices", boundary_state_indices),
                            ("boundary_recovery_lens", boundary_recovery_lens)):
                if t is not None:
                    _need(t, name, torch.int32, dev, 1)
                    if t.shape[0] < B or not t.is_contiguous():
                        raise ValueError(f"{name} must be contiguous with at least B entries")
            align = AlignArgs()
            align.final_state_indices = _ptr(final_state_indices)
            align.boundary_state_indices = _ptr(boundary_state_indices)
            align.boundary_recovery_lens = _ptr(boundary_recovery_lens)
        a = CommitArgs()
        a.L, a.B, a.H, a.K, a.V, a.Q = self.L, B, self.H, self.K, self.V, self.window
        a.null_block_id = null_block_id
        a.num_slots, a.num_record_rows = self.slots, self.rows
        a.state_base, a.state_slot_stride = self.state_base.data_ptr(), self.state_stride.data_ptr()
        a.corr_base, a.corr_row_stride = self.corr_base.data_ptr(), self.corr_stride.data_ptr()
        a.kg_base, a.kg_row_stride = self.kg_base.data_ptr(), self.kg_stride.data_ptr()
        a.A_log, a.dt_bias = self.A_log.data_ptr(), self.dt_bias.data_ptr()
        a.gate_mode = GATE_SOFTPLUS if self.lower_bound is None else GATE_LOWER_BOUND
        a.lower_bound = 0.0 if self.lower_bound is None else float(self.lower_bound)
        a.query_start_loc, a.state_indices = query_start_loc.data_ptr(), state_indices.data_ptr()
        a.record_indices = _ptr(record_indices)
        a.num_accepted = num_accepted_tokens.data_ptr()
        a.workspace = _ptr(workspace)
        handle = ctypes.c_void_p(_stream_handle(dev, stream))
        if align is None:
            _check(load_library().kda_commit(ctypes.byref(a), handle))
        else:
            _check(load_library().kda_commit_align(ctypes.byref(a), ctypes.byref(align), handle))


NOALLOC_MAX_LAYERS = 64  # KDA_NOALLOC_MAX_LAYERS


def commit_noalloc(*, states: Sequence[torch.Tensor], corrections: Sequence[torch.Tensor],
                   key_gates: Sequence[torch.Tensor], A_log: torch.Tensor, dt_bias: torch.Tensor,
                   lower_bound: float | None, window: int, num_accepted_tokens: torch.Tensor,
                   state_indices: torch.Tensor, query_start_loc: torch.Tensor,
                   record_indices: torch.Tensor | None = None, null_block_id: int = 0,
                   workspace: torch.Tensor | None = None, stream=None) -> None:
    """The commit of ``CommitContext.commit`` through kda_commit_noalloc: the
    per-layer tables stay on the host and the library copies them into its
    static device scratch (at most NOALLOC_MAX_LAYERS layers), so neither this
    function nor the library allocates device memory.  Calls that can overlap
    on the device race on that scratch; the first call on a device does the
    scratch set-up and belongs before any stream capture."""
    L = len(states)
    if L == 0 or not (L == len(corrections) == len(key_gates)):
        raise ValueError("states, corrections and key_gates need one entry per layer")
    ref = states[0]
    dev = ref.device
    slots, H, V, K = ref.shape
    rows = corrections[0].shape[0]
    for l in range(L):
        _need(states[l], f"states[{l}]", torch.float32, dev, 4)
        _need(corrections[l], f"corrections[{l}]", torch.float32, dev, 4)
        _need(key_gates[l], f"key_gates[{l}]", torch.bfloat16, dev, 4)
        if states[l].shape != ref.shape:
            raise ValueError("layers need matching state shapes")
        if corrections[l].shape != (rows, H, window, V) or key_gates[l].shape != (rows, H, window, 2 * K):
            raise ValueError("layers need matching record shapes")
        _inner_contiguous(states[l], f"states[{l}]", 3)
        _inner_contiguous(corrections[l], f"corrections[{l}]", 3)
        _inner_contiguous(key_gates[l], f"key_gates[{l}]", 3)
    _need(A_log, "A_log", torch.float32, dev)
    _need(dt_bias, "dt_bias", torch.float32, dev)
    if A_log.numel() != L * H or dt_bias.numel() != L * H * K:
        raise ValueError("A_log must be [L, H] and dt_bias [L, H*K]")
    if not (A_log.is_contiguous() and dt_bias.is_contiguous()):
        raise ValueError("A_log and dt_bias must be contiguous")
    B = state_indices.shape[0]
    for name, t in (("num_accepted_tokens", num_accepted_tokens), ("state_indices", state_indices),
                    ("query_start_loc", query_start_loc)):
        _need(t, name, torch.int32, dev, 1)
        if not t.is_contiguous():
            raise ValueError("commit metadata must be contiguous")
    if query_start_loc.shape[0] != B + 1 or num_accepted_tokens.shape[0] < B:
        raise ValueError("commit metadata is incompatible: query_start_loc [B+1], num_accepted [B]")
    if record_indices is not None:
        _need(record_indices, "record_indices", torch.int32, dev, 1)
        if record_indices.shape[0] < B or not record_indices.is_contiguous():
            raise ValueError("record_indices is too short")
    if workspace is not None:
        _need(workspace, "workspace", torch.int32, dev)

    def host_table(vals):
        return (ctypes.c_int64 * L)(*vals)

    tables = [host_table([t.data_ptr() for t in states]), host_table([t.stride(0) for t in states]),
              host_table([t.data_ptr() for t in corrections]), host_table([t.stride(0) for t in corrections]),
              host_table([t.data_ptr() for t in key_gates]), host_table([t.stride(0) for t in key_gates])]
    a = CommitArgs()
    a.L, a.B, a.H, a.K, a.V, a.Q = L, B, H, K, V, window
    a.null_block_id = null_block_id
    a.num_slots, a.num_record_rows = slots, rows
    a.state_base, a.state_slot_stride, a.corr_base, a.corr_row_stride, a.kg_base, a.kg_row_stride = (
        ctypes.cast(t, ctypes.c_void_p).value for t in tables)
    a.A_log, a.dt_bias = A_log.data_ptr(), dt_bias.data_ptr()
    a.gate_mode = GATE_SOFTPLUS if lower_bound is None else GATE_LOWER_BOUND
    a.lower_bound = 0.0 if lower_bound is None else float(lower_bound)
    a.query_start_loc, a.state_indices = query_start_loc.data_ptr(), state_indices.data_ptr()
    a.record_indices = _ptr(record_indices)
    a.num_accepted = num_accepted_tokens.data_ptr()
    a.workspace = _ptr(workspace)
    _check(load_library().kda_commit_noalloc(ctypes.byref(a), ctypes.c_void_p(_stream_handle(dev, stream))))
