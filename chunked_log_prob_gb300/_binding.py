"""ctypes binding of the C ABI in include/grpo_gb300.h (argument marshalling only).

Every step of the computation runs in the CUDA library; this module only
checks tensors, passes their device pointers and the current CUDA stream, and
turns error codes into exceptions. There is no CPU path: if the library is not
built, importing the package raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB_PATH

GRPO_OK = 0
GRPO_ERR_DEVICE_TIMEOUT = -7
GRPO_ERR_BAD_TOKEN_ID = -8
GRPO_ERR_NONFINITE = -9
STATUS_NAMES = {
    0: "GRPO_OK", -1: "GRPO_ERR_INVALID_ARG", -2: "GRPO_ERR_MISALIGNED",
    -3: "GRPO_ERR_UNSUPPORTED_SHAPE", -4: "GRPO_ERR_WORKSPACE_TOO_SMALL",
    -5: "GRPO_ERR_UNSUPPORTED_DEVICE", -6: "GRPO_ERR_CUDA",
    -7: "GRPO_ERR_DEVICE_TIMEOUT", -8: "GRPO_ERR_BAD_TOKEN_ID", -9: "GRPO_ERR_NONFINITE",
}


class GrpoShape(ctypes.Structure):
    _fields_ = [("n_tokens", ctypes.c_int64), ("seq_len", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class GrpoParams(ctypes.Structure):
    _fields_ = [("eps_low", ctypes.c_float), ("eps_high", ctypes.c_float),
                ("beta", ctypes.c_float), ("loss_denominator", ctypes.c_float),
                ("chunk_tokens", ctypes.c_int32), ("vocab_block", ctypes.c_int32),
                ("flags", ctypes.c_uint32), ("raster_rows", ctypes.c_int32),
                ("logit_scale_multiply", ctypes.c_float), ("logit_scale_divide", ctypes.c_float),
                ("logit_softcapping", ctypes.c_float), ("temperature", ctypes.c_float),
                ("workspace_limit_bytes", ctypes.c_uint64)]


class GrpoPlanInfo(ctypes.Structure):
    _fields_ = [("chunk_rows", ctypes.c_int32), ("vocab_block", ctypes.c_int32),
                ("n_chunks", ctypes.c_int32), ("n_vocab_blocks", ctypes.c_int32),
                ("fwd_splits", ctypes.c_int32), ("launches_logp", ctypes.c_int32),
                ("launches_loss", ctypes.c_int32), ("g_in_dh_gemm", ctypes.c_int32),
                ("stored_logits", ctypes.c_int32), ("single_pass", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_uint64)]


class GrpoError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({status_string(code)})")


class GrpoKernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 40), ("launches", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("total_ms", ctypes.c_double)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    P = ctypes.POINTER
    lib.grpo_default_params.argtypes = [P(GrpoParams)]
    lib.grpo_default_params.restype = None
    lib.grpo_workspace_size.argtypes = [P(GrpoShape), P(GrpoParams), P(sz)]
    lib.grpo_workspace_size.restype = ctypes.c_int
    lib.grpo_logp_fwd.argtypes = [vp, vp, vp, vp, vp, P(GrpoShape), P(GrpoParams), vp, sz, vp]
    lib.grpo_logp_fwd.restype = ctypes.c_int
    lib.grpo_loss_fwd_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      P(GrpoShape), P(GrpoParams), vp, sz, vp]
    lib.grpo_loss_fwd_bwd.restype = ctypes.c_int
    lib.grpo_get_plan.argtypes = [P(GrpoShape), P(GrpoParams), P(GrpoPlanInfo)]
    lib.grpo_get_plan.restype = ctypes.c_int
    lib.grpo_read_device_status.argtypes = [vp, P(ctypes.c_int), vp]
    lib.grpo_read_device_status.restype = ctypes.c_int
    lib.grpo_logp_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, P(GrpoShape), vp]
    lib.grpo_logp_fwd_noalloc.restype = ctypes.c_int
    lib.grpo_selftest_bounded_wait.argtypes = [vp, sz, vp]
    lib.grpo_selftest_bounded_wait.restype = ctypes.c_int
    lib.grpo_launch_timing_enable.argtypes = [ctypes.c_int]
    lib.grpo_launch_timing_enable.restype = ctypes.c_int
    lib.grpo_launch_timing_read.argtypes = [P(GrpoKernelTime), ctypes.c_int, P(ctypes.c_int)]
    lib.grpo_launch_timing_read.restype = ctypes.c_int
    lib.grpo_status_string.argtypes = [ctypes.c_int]
    lib.grpo_status_string.restype = ctypes.c_char_p
    return lib


lib = _load()

EXPORTED = ("grpo_default_params", "grpo_workspace_size", "grpo_logp_fwd",
            "grpo_loss_fwd_bwd", "grpo_get_plan", "grpo_read_device_status",
            "grpo_logp_fwd_noalloc", "grpo_selftest_bounded_wait", "grpo_launch_timing_enable",
            "grpo_launch_timing_read", "grpo_status_string")

FLAG_STORED_LOGITS = 1
FLAG_SINGLE_CTA = 2
FLAG_SEQUENCE_MEAN = 4
FLAG_FIT_FREE_MEMORY = 8
FLAG_RECOMPUTE_LOGITS = 16
FLAG_SINGLE_PASS = 32

# Largest batch of the workspace-free forward (its static device scratch).
NOALLOC_MAX_TOKENS = 8192


def status_string(code: int) -> str:
    return lib.grpo_status_string(int(code)).decode()


def make_params(eps_low=0.2, eps_high=0.2, beta=0.001, loss_denominator=0.0,
                chunk_tokens=0, vocab_block=0, *, logit_scale_multiply=0.0,
                logit_scale_divide=0.0, logit_softcapping=0.0, temperature=0.0,
                flags=0, workspace_limit_bytes=0, raster_rows=0) -> GrpoParams:
    p = GrpoParams()
    lib.grpo_default_params(ctypes.byref(p))
    p.eps_low, p.eps_high, p.beta = eps_low, eps_high, beta
    p.loss_denominator = loss_denominator
    p.chunk_tokens, p.vocab_block = chunk_tokens, vocab_block
    p.logit_scale_multiply, p.logit_scale_divide = logit_scale_multiply, logit_scale_divide
    p.logit_softcapping, p.temperature = logit_softcapping, temperature
    p.flags = flags
    p.workspace_limit_bytes = int(workspace_limit_bytes)
    p.raster_rows = int(raster_rows)
    return p


def make_shape(n_tokens, seq_len, hidden, vocab) -> GrpoShape:
    return GrpoShape(int(n_tokens), int(seq_len), int(hidden), int(vocab), 0)


def grpo_workspace_size(n_tokens, hidden, vocab, seq_len=1, params: GrpoParams | None = None) -> int:
    out = ctypes.c_size_t(0)
    shape = make_shape(n_tokens, seq_len, hidden, vocab)
    rc = lib.grpo_workspace_size(ctypes.byref(shape),
                                 ctypes.byref(params) if params is not None else None,
                                 ctypes.byref(out))
    if rc != GRPO_OK:
        raise GrpoError(rc, "grpo_workspace_size")
    return int(out.value)


def grpo_get_plan(n_tokens, hidden, vocab, seq_len=1, params: GrpoParams | None = None) -> dict:
    """The chunking and launch count a call would use on the current device."""
    info = GrpoPlanInfo()
    shape = make_shape(n_tokens, seq_len, hidden, vocab)
    rc = lib.grpo_get_plan(ctypes.byref(shape),
                           ctypes.byref(params) if params is not None else None,
                           ctypes.byref(info))
    if rc != GRPO_OK:
        raise GrpoError(rc, "grpo_get_plan")
    return {name: int(getattr(info, name)) for name, _ in GrpoPlanInfo._fields_
            if name != "reserved"}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t, name, dtype, shape, device):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def alloc_workspace(n_tokens, hidden, vocab, seq_len=1, params=None, device=None) -> torch.Tensor:
    nbytes = grpo_workspace_size(n_tokens, hidden, vocab, seq_len, params)
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def grpo_logp_fwd(hidden, W, ids, *, params: GrpoParams | None = None, workspace=None,
                  logp=None, lse=None, want_lse=False):
    """logp[t] = h_t . W[ids[t]] - logsumexp_v h_t . W_v (fp32), on hidden's device."""
    dev = hidden.device
    N, D = hidden.shape
    V = W.shape[0]
    _check(hidden, "hidden", torch.bfloat16, (N, D), dev)
    _check(W, "W", torch.bfloat16, (V, D), dev)
    _check(ids, "ids", torch.int32, (N,), dev)
    if logp is None:
        logp = torch.empty(N, dtype=torch.float32, device=dev)
    if want_lse and lse is None:
        lse = torch.empty(N, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(N, D, V, 1, params, dev)
    shape = make_shape(N, 1, D, V)
    rc = lib.grpo_logp_fwd(_ptr(hidden), _ptr(W), _ptr(ids), _ptr(logp), _ptr(lse),
                           ctypes.byref(shape),
                           ctypes.byref(params) if params is not None else None,
                           _ptr(workspace), workspace.numel(), _stream(dev))
    if rc != GRPO_OK:
        raise GrpoError(rc, "grpo_logp_fwd")
    return logp, lse


def grpo_loss_fwd_bwd(hidden, W, ids, mask, old_logp, ref_logp, adv, seq_len, *,
                      params: GrpoParams | None = None, workspace=None, want_logp=True,
                      loss=None, logp=None, dH=None, dW=None, want_dW=False):
    """Fused GRPO loss forward + backward to hidden (and to the lm_head weight).

    Returns (loss[1], logp[N] | None, dH[N, D]) or, with want_dW / dW given,
    (loss, logp, dH, dW[V, D] fp32).
    """
    dev = hidden.device
    N, D = hidden.shape
    V = W.shape[0]
    _check(hidden, "hidden", torch.bfloat16, (N, D), dev)
    _check(W, "W", torch.bfloat16, (V, D), dev)
    _check(ids, "ids", torch.int32, (N,), dev)
    if mask is not None:
        _check(mask, "mask", torch.uint8, (N,), dev)
    _check(old_logp, "old_logp", torch.float32, (N,), dev)
    _check(ref_logp, "ref_logp", torch.float32, (N,), dev)
    if seq_len <= 0 or N % seq_len != 0:
        raise ValueError("n_tokens must be a multiple of seq_len")
    _check(adv, "adv", torch.float32, (N // seq_len,), dev)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=dev)
    if want_logp and logp is None:
        logp = torch.empty(N, dtype=torch.float32, device=dev)
    if dH is None:
        dH = torch.empty(N, D, dtype=torch.bfloat16, device=dev)
    if want_dW and dW is None:
        dW = torch.empty(V, D, dtype=torch.float32, device=dev)
    if dW is not None:
        _check(dW, "dW", torch.float32, (V, D), dev)
    if workspace is None:
        workspace = alloc_workspace(N, D, V, seq_len, params, dev)
    shape = make_shape(N, seq_len, D, V)
    rc = lib.grpo_loss_fwd_bwd(_ptr(hidden), _ptr(W), _ptr(ids), _ptr(mask), _ptr(old_logp),
                               _ptr(ref_logp), _ptr(adv), _ptr(loss), _ptr(logp), _ptr(dH),
                               _ptr(dW), ctypes.byref(shape),
                               ctypes.byref(params) if params is not None else None,
                               _ptr(workspace), workspace.numel(), _stream(dev))
    if rc != GRPO_OK:
        raise GrpoError(rc, "grpo_loss_fwd_bwd")
    if dW is not None:
        return loss, logp, dH, dW
    return loss, logp, dH


def grpo_read_device_status(workspace) -> int:
    st = ctypes.c_int(0)
    rc = lib.grpo_read_device_status(_ptr(workspace), ctypes.byref(st),
                                     _stream(workspace.device))
    if rc != GRPO_OK:
        raise GrpoError(rc, "grpo_read_device_status")
    return int(st.value)


def grpo_logp_fwd_noalloc(hidden, W, ids, logp, lse=None):
    """Workspace-free forward for callers that cannot allocate device memory.

    Same results as grpo_logp_fwd; scratch is a static device array inside the
    library (n_tokens <= NOALLOC_MAX_TOKENS). The caller passes the outputs.
    Calls that overlap on the GPU race on the shared scratch.
    """
    dev = hidden.device
    N, D = hidden.shape
    V = W.shape[0]
    _check(hidden, "hidden", torch.bfloat16, (N, D), dev)
    _check(W, "W", torch.bfloat16, (V, D), dev)
    _check(ids, "ids", torch.int32, (N,), dev)
    _check(logp, "logp", torch.float32, (N,), dev)
    if lse is not None:
        _check(lse, "lse", torch.float32, (N,), dev)
    shape = make_shape(N, 1, D, V)
    rc = lib.grpo_logp_fwd_noalloc(_ptr(hidden), _ptr(W), _ptr(ids), _ptr(logp), _ptr(lse),
                                   ctypes.byref(shape), _stream(dev))
    if rc != GRPO_OK:
        raise GrpoError(rc, "grpo_logp_fwd_noalloc")
    return logp, lse


def grpo_selftest_bounded_wait(workspace) -> int:
    """Runs the bounded-wait self-test; returns the device status it left (-7 expected)."""
    rc = lib.grpo_selftest_bounded_wait(_ptr(workspace), workspace.numel(),
                                        _stream(workspace.device))
    if rc != GRPO_OK:
        raise GrpoError(rc, "grpo_selftest_bounded_wait")
    return grpo_read_device_status(workspace)


def grpo_launch_timing_enable(on: bool = True) -> None:
    """Per-launch CUDA-event timing for the calling thread (off by default)."""
    rc = lib.grpo_launch_timing_enable(1 if on else 0)
    if rc != GRPO_OK:
        raise GrpoError(rc, "grpo_launch_timing_enable")


def grpo_launch_timing_read(capacity: int = 64) -> list[dict]:
    """Waits for the timed launches, returns and clears their per-kernel sums:
    ``[{"name", "launches", "total_ms"}]`` in order of first launch."""
    buf = (GrpoKernelTime * capacity)()
    count = ctypes.c_int(0)
    rc = lib.grpo_launch_timing_read(buf, int(capacity), ctypes.byref(count))
    if rc != GRPO_OK:
        raise GrpoError(rc, "grpo_launch_timing_read")
    if count.value > capacity:
        raise GrpoError(-1, f"grpo_launch_timing_read: {count.value} kernels > capacity {capacity}")
    return [{"name": buf[i].name.decode(), "launches": int(buf[i].launches),
             "total_ms": float(buf[i].total_ms)} for i in range(count.value)]
