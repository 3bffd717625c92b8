"""ctypes binding to libsanta.so (the C ABI in include/santa.h).

Argument marshalling only: every step of the decode step runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  If the library has not been built
or cannot be loaded, every call raises -- there is no CPU path.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsanta.so")

OK = 0
DENSE, STRATIFIED, SYSTEMATIC, IID = 0, 1, 2, 3
MODES = {"dense": DENSE, "stratified": STRATIFIED, "systematic": SYSTEMATIC, "iid": IID}
GROUP_DEDUP = 0x100  # or-ed into a sampling mode: V rows loaded once per KV-head group
OUT_BF16 = 0x200     # or-ed into any mode: out is bf16 (the fp32 result rounded once)
BERNOULLI_QK = 0x400  # or-ed into any mode: score with each head's ternary query draw
TWO_PASS = 0x800      # or-ed into a sampling mode: never the single-pass cluster kernel
DEV_BAD_SEQLEN, DEV_TIMEOUT = 1, 2

# every symbol include/santa.h declares
EXPORTS = ("santa_workspace_size", "santa_workspace_init", "santa_decode", "santa_sample_points",
           "santa_device_status", "santa_status_string", "santa_version", "santa_decode_static",
           "santa_set_wait_limit", "santa_ternary_query", "santa_call_info", "santa_timeline_buffer")
ERR_DEVICE = -6
ERR_SCRATCH = -7
STATIC_SCRATCH_BYTES = 16 << 20


class SantaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("n_max", ctypes.c_int32), ("scale", ctypes.c_float)]


_lock = threading.Lock()
_lib = None
_lib_path = None


def load(path: str | None = None):
    """Load libsanta.so (raises if it is missing: build it with __graft_entry__.build()).
    The SANTA_LIBRARY environment variable, if set, names another build to load; so does
    `path`, on the first call of a process (one build per process)."""
    global _lib, _lib_path
    with _lock:
        if _lib is not None:
            if path is not None and os.path.realpath(path) != _lib_path:
                raise RuntimeError(f"{_lib_path} is loaded already; one libsanta build per process")
            return _lib
        p = path or os.environ.get("SANTA_LIBRARY", LIB_PATH)
        if not os.path.exists(p):
            raise RuntimeError(f"libsanta.so not found at {p}; build it first (python -c "
                               "'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        vp, i32, u64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint64, ctypes.c_size_t
        lib.santa_workspace_size.argtypes = [ctypes.POINTER(Shape), i32, i32, ctypes.POINTER(sz)]
        lib.santa_workspace_size.restype = ctypes.c_int
        lib.santa_workspace_init.argtypes = [vp, sz, vp]
        lib.santa_workspace_init.restype = ctypes.c_int
        lib.santa_decode.argtypes = [ctypes.POINTER(Shape), vp, vp, vp, vp, i32, i32, u64, vp, vp, vp, sz, vp]
        lib.santa_decode.restype = ctypes.c_int
        lib.santa_sample_points.argtypes = [i32, i32, i32, i32, u64, vp, vp]
        lib.santa_sample_points.restype = ctypes.c_int
        lib.santa_device_status.argtypes = [vp, ctypes.POINTER(i32), vp]
        lib.santa_device_status.restype = ctypes.c_int
        lib.santa_status_string.argtypes = [ctypes.c_int]
        lib.santa_status_string.restype = ctypes.c_char_p
        lib.santa_decode_static.argtypes = [ctypes.POINTER(Shape), vp, vp, vp, vp, i32, i32, u64, vp, vp, vp]
        lib.santa_decode_static.restype = ctypes.c_int
        lib.santa_ternary_query.argtypes = [i32, i32, i32, vp, u64, vp, vp]
        lib.santa_ternary_query.restype = ctypes.c_int
        lib.santa_call_info.argtypes = [ctypes.POINTER(Shape), i32, i32, ctypes.POINTER(i32)]
        lib.santa_call_info.restype = ctypes.c_int
        lib.santa_timeline_buffer.argtypes = [vp, sz]
        lib.santa_timeline_buffer.restype = ctypes.c_int
        lib.santa_set_wait_limit.argtypes = [u64]
        lib.santa_set_wait_limit.restype = ctypes.c_int
        lib.santa_version.argtypes = []
        lib.santa_version.restype = ctypes.c_int
        _lib, _lib_path = lib, os.path.realpath(p)
        return lib


def status_string(status: int) -> str:
    return load().santa_status_string(int(status)).decode()


def _check(rc: int, what: str):
    if rc != OK:
        raise SantaError(rc, what)


def _mode(mode) -> int:
    return MODES[mode] if isinstance(mode, str) else int(mode)


def make_shape(B, H_q, H_kv, d, n_max, scale: float = 0.0) -> Shape:
    return Shape(int(B), int(H_q), int(H_kv), int(d), int(n_max), float(scale))


def workspace_size(shape: Shape, S: int, mode) -> int:
    n = ctypes.c_size_t(0)
    _check(load().santa_workspace_size(ctypes.byref(shape), int(S), _mode(mode), ctypes.byref(n)),
           "santa_workspace_size")
    return int(n.value)


def _stream_ptr(stream) -> int | None:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def new_workspace(nbytes: int, device, stream=None) -> torch.Tensor:
    """A zero-initialised workspace (torch allocation, 256-byte aligned)."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    _check(load().santa_workspace_init(ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                                       ctypes.c_void_p(_stream_ptr(stream))), "santa_workspace_init")
    return ws


_ws_cache: dict = {}


def _cached_workspace(nbytes: int, device, stream) -> torch.Tensor:
    key = (torch.device(device), _stream_ptr(stream))
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = new_workspace(nbytes, device, stream)
        _ws_cache[key] = ws
    return ws


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, seq_lens: torch.Tensor,
           S: int, mode="systematic", seed: int = 0, scale: float = 0.0, out: torch.Tensor | None = None,
           idx_out: torch.Tensor | None = None, want_idx: bool = True, workspace: torch.Tensor | None = None,
           stream=None, group_dedup: bool = False, out_dtype: torch.dtype = torch.float32,
           bernoulli: bool = False, two_pass: bool = False):
    """One SANTA (or dense) decode step on the GPU.  q [B,H_q,d], k/v [B,H_kv,n_max,d] bf16,
    seq_lens [B] int32, all on one CUDA device.  Returns (out [B,H_q,d], idx int32
    [B,H_q,S] or None).  out is fp32, or bf16 (SANTA_OUT_BF16) when `out` is a bf16 tensor
    or out_dtype is torch.bfloat16.  group_dedup: load each sampled V row once per group of
    query heads sharing a KV head (SANTA_GROUP_DEDUP).  bernoulli: score with each head's
    ternary query draw (SANTA_BERNOULLI_QK).  two_pass: the score and value stages as two
    launches even where the single-pass cluster kernel applies (SANTA_TWO_PASS)."""
    m = _mode(mode)
    B, H_q, d = q.shape
    _, H_kv, n_max, d2 = k_cache.shape
    for t, name in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if seq_lens.dtype != torch.int32 or not seq_lens.is_cuda:
        raise ValueError("seq_lens must be an int32 CUDA tensor")
    if v_cache.shape != k_cache.shape or d2 != d:
        raise ValueError("k_cache/v_cache/q shapes disagree")
    shape = make_shape(B, H_q, H_kv, d, n_max, scale)
    dev = q.device
    if out is None:
        out = torch.empty(B, H_q, d, dtype=out_dtype, device=dev)
    if out.dtype not in (torch.float32, torch.bfloat16) or not out.is_contiguous() or out.shape != (B, H_q, d):
        raise ValueError("out must be a contiguous fp32 or bf16 [B, H_q, d] tensor")
    if m != DENSE and want_idx and idx_out is None:
        idx_out = torch.empty(B, H_q, S, dtype=torch.int32, device=dev)
    nbytes = workspace_size(shape, S if m != DENSE else 1, m)
    ws = workspace if workspace is not None else _cached_workspace(nbytes, dev, stream)
    mf = m | (GROUP_DEDUP if (group_dedup and m != DENSE) else 0) | (OUT_BF16 if out.dtype == torch.bfloat16 else 0) \
        | (BERNOULLI_QK if bernoulli else 0) | (TWO_PASS if (two_pass and m != DENSE) else 0)
    rc = load().santa_decode(ctypes.byref(shape), ctypes.c_void_p(q.data_ptr()),
                             ctypes.c_void_p(k_cache.data_ptr()), ctypes.c_void_p(v_cache.data_ptr()),
                             ctypes.c_void_p(seq_lens.data_ptr()), int(S), mf, ctypes.c_uint64(seed),
                             ctypes.c_void_p(out.data_ptr()),
                             ctypes.c_void_p(idx_out.data_ptr() if (idx_out is not None and m != DENSE) else 0),
                             ctypes.c_void_p(ws.data_ptr()), ws.numel(), ctypes.c_void_p(_stream_ptr(stream)))
    _check(rc, "santa_decode")
    return out, (idx_out if m != DENSE else None)


class DecodePlan:
    """santa_decode with every argument but the seed marshalled once: the checks of
    decode(), the shape, the workspace and the ctypes arguments are built in the
    constructor, and each call is one foreign call.  For decode loops where the tensors
    stay put (the call reads whatever the tensors hold at that time)."""

    def __init__(self, q, k_cache, v_cache, seq_lens, S: int, mode="systematic", scale: float = 0.0,
                 out: torch.Tensor | None = None, idx_out: torch.Tensor | None = None, want_idx: bool = True,
                 workspace: torch.Tensor | None = None, stream=None, group_dedup: bool = False,
                 out_dtype: torch.dtype = torch.float32, bernoulli: bool = False, two_pass: bool = False):
        m = _mode(mode)
        # one checked call through decode() fixes every buffer (and runs the step once)
        self.out, self.idx_out = decode(q, k_cache, v_cache, seq_lens, S, m, 0, scale, out, idx_out, want_idx,
                                        workspace, stream, group_dedup, out_dtype, bernoulli, two_pass)
        B, H_q, d = q.shape
        _, H_kv, n_max, _ = k_cache.shape
        self._shape = make_shape(B, H_q, H_kv, d, n_max, scale)
        nbytes = workspace_size(self._shape, S if m != DENSE else 1, m)
        ws = workspace if workspace is not None else _cached_workspace(nbytes, q.device, stream)
        # the buffers (and the stream object, if one was given) stay alive with the plan
        self._keep = (q, k_cache, v_cache, seq_lens, ws, stream)
        flags = m | (GROUP_DEDUP if (group_dedup and m != DENSE) else 0) | \
            (OUT_BF16 if self.out.dtype == torch.bfloat16 else 0) | (BERNOULLI_QK if bernoulli else 0) | \
            (TWO_PASS if (two_pass and m != DENSE) else 0)
        vp = ctypes.c_void_p
        self._fn = load().santa_decode
        self._pre = (ctypes.byref(self._shape), vp(q.data_ptr()), vp(k_cache.data_ptr()), vp(v_cache.data_ptr()),
                     vp(seq_lens.data_ptr()), int(S), flags)
        self._post = (vp(self.out.data_ptr()),
                      vp(self.idx_out.data_ptr() if (self.idx_out is not None and m != DENSE) else 0),
                      vp(ws.data_ptr()), ws.numel(), vp(_stream_ptr(stream)))

    def __call__(self, seed: int):
        rc = self._fn(*self._pre, ctypes.c_uint64(seed), *self._post)
        if rc != 0:
            _check(rc, "santa_decode")
        return self.out, self.idx_out


def call_info(shape: Shape, S: int, mode, group_dedup: bool = False, bernoulli: bool = False,
              two_pass: bool = False) -> int:
    """santa_call_info: the kernel launches one decode call with this shape, S and mode
    enqueues on the current device (1: the single-pass cluster kernel)."""
    m = _mode(mode) | (GROUP_DEDUP if group_dedup else 0) | (BERNOULLI_QK if bernoulli else 0) | \
        (TWO_PASS if two_pass else 0)
    n = ctypes.c_int32(0)
    _check(load().santa_call_info(ctypes.byref(shape), int(S), m, ctypes.byref(n)), "santa_call_info")
    return int(n.value)


def set_wait_limit(limit_ns: int) -> None:
    """santa_set_wait_limit: how long a kernel's pipeline waits may last before it gives
    up with SANTA_DEV_TIMEOUT (0: the default of 2 s).  A diagnostic knob."""
    _check(load().santa_set_wait_limit(ctypes.c_uint64(int(limit_ns))), "santa_set_wait_limit")


def sample_points(B: int, H_q: int, S: int, mode, seed: int, device="cuda", stream=None) -> torch.Tensor:
    t = torch.empty(B, H_q, S, dtype=torch.float64, device=device)
    _check(load().santa_sample_points(int(B), int(H_q), int(S), _mode(mode), ctypes.c_uint64(seed),
                                      ctypes.c_void_p(t.data_ptr()), ctypes.c_void_p(_stream_ptr(stream))),
           "santa_sample_points")
    return t


def ternary_query(q: torch.Tensor, seed: int, stream=None) -> torch.Tensor:
    """santa_ternary_query: each head's Bernoulli qK^T draw (bf16 [B,H_q,d])."""
    if q.dtype != torch.bfloat16 or not q.is_cuda or not q.is_contiguous() or q.dim() != 3:
        raise ValueError("q must be a contiguous bf16 CUDA tensor [B, H_q, d]")
    B, H_q, d = q.shape
    out = torch.empty_like(q)
    _check(load().santa_ternary_query(int(B), int(H_q), int(d), ctypes.c_void_p(q.data_ptr()), ctypes.c_uint64(seed),
                                      ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(_stream_ptr(stream))),
           "santa_ternary_query")
    return out


def device_status(workspace: torch.Tensor | None, stream=None) -> int:
    """santa_device_status: the device error word of `workspace` (None: the static scratch
    of santa_decode_static on the current device), read and cleared."""
    code = ctypes.c_int32(0)
    rc = load().santa_device_status(ctypes.c_void_p(workspace.data_ptr() if workspace is not None else 0),
                                    ctypes.byref(code), ctypes.c_void_p(_stream_ptr(stream)))
    if rc not in (OK, ERR_DEVICE):
        _check(rc, "santa_device_status")
    return int(code.value)
