"""TEST INFRASTRUCTURE ONLY: ctypes wrapper around the fp64 CPU oracle (santa_oracle.c).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The CUDA library never links, loads or calls it, and this wrapper
does argument marshalling only: every step of the oracle's arithmetic is in the C file,
which cites the passages of "Stochastic Sparse Attention for Memory-Bound Inference"
(abstract) that it follows.

Mode numbers (the oracle's own constants): 0 dense, 1 stratified, 2 systematic, 3 iid.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "santa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libsanta_oracle.so")

DENSE, STRATIFIED, SYSTEMATIC, IID = 0, 1, 2, 3
MODES = {"dense": DENSE, "stratified": STRATIFIED, "systematic": SYSTEMATIC, "iid": IID}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile santa_oracle.c with gcc (-O2, OpenMP, no machine-specific flags)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i32, u64, f32 = ctypes.c_int32, ctypes.c_uint64, ctypes.c_float
        vp = ctypes.c_void_p
        lib.oracle_philox4x64_10.argtypes = [vp, vp, vp]
        lib.oracle_philox4x64_10.restype = None
        lib.oracle_points.argtypes = [ctypes.c_int, i32, u64, i32, i32, vp]
        lib.oracle_points.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [i32, i32, i32, i32, i32, f32, vp, vp, vp, vp, i32,
                                      ctypes.c_int, u64, ctypes.c_int, vp, vp, i32, vp, vp, vp]
        lib.oracle_ternary_query.argtypes = [i32, vp, u64, i32, i32, vp]
        lib.oracle_ternary_query.restype = i32
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_cdf.argtypes = [i32, i32, i32, i32, i32, f32, vp, vp, vp, i32, i32, vp, vp]
        lib.oracle_cdf.restype = ctypes.c_int
        lib.oracle_gather.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, i32, vp]
        lib.oracle_gather.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(x) -> np.ndarray:
    """bf16 bit patterns as a contiguous uint16 array (accepts a torch bf16 tensor or a
    uint16 numpy array)."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype == torch.bfloat16, x.dtype
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def philox4x64_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint64).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint64).reshape(2))
    out = np.zeros(4, dtype=np.uint64)
    _load().oracle_philox4x64_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def points(mode, S: int, seed: int, b: int, h: int) -> np.ndarray:
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    t = np.zeros(S, dtype=np.float64)
    if _load().oracle_points(m, S, seed, b, h, _ptr(t)) != 0:
        raise ValueError("oracle_points: bad mode or S")
    return t


def ternary_query(q, seed: int):
    """Bernoulli qK^T: the ternary draw of every query head, as a bf16 torch tensor
    [B,H_q,d] (values -a, 0, +a with a = max |q| of the head), and the count of non-zero
    features per head (int32 [B,H_q])."""
    import torch
    qb = _bits(q)
    B, H_q, d = qb.shape
    qt = np.zeros_like(qb)
    nnz = np.zeros((B, H_q), dtype=np.int32)
    lib = _load()
    for b in range(B):
        for h in range(H_q):
            row = np.ascontiguousarray(qb[b, h])
            out = np.zeros(d, dtype=np.uint16)
            nnz[b, h] = lib.oracle_ternary_query(d, _ptr(row), seed, b, h, _ptr(out))
            qt[b, h] = out
    return torch.from_numpy(qt.view(np.int16)).view(torch.bfloat16), nnz


def decode(q, k, v, seq_lens, S: int, mode, seed: int = 0, scale: float | None = None,
           t=None, pairs=None, want_idx: bool = True, want_Z: bool = False, bernoulli: bool = False):
    """Oracle decode step.  q [B,H_q,d], k/v [B,H_kv,n_max,d] (bf16 torch tensors or
    uint16 bit arrays), seq_lens [B] int.  bernoulli: score with each head's ternary
    query draw (Bernoulli qK^T, seeded by `seed`).  Returns (out fp64 [B,H_q,d], idx
    int32 [B,H_q,S] or None[, Z fp64 [B,H_q]])."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, H_q, d = qb.shape
    _, H_kv, n_max, d2 = kb.shape
    assert d2 == d and vb.shape == kb.shape
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(B))
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(d)))
    out = np.zeros((B, H_q, d), dtype=np.float64)
    idx = np.zeros((B, H_q, S), dtype=np.int32) if (want_idx and m != DENSE) else None
    Z = np.zeros((B, H_q), dtype=np.float64) if want_Z else None
    tt = None if t is None else np.ascontiguousarray(np.asarray(t, dtype=np.float64).reshape(B, H_q, S))
    pr = None
    npairs = 0
    if pairs is not None:
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        npairs = pr.shape[0]
    rc = _load().oracle_decode(B, H_q, H_kv, d, n_max, ctypes.c_float(scale), _ptr(qb), _ptr(kb),
                               _ptr(vb), _ptr(sl), S if m != DENSE else 0, m, seed, 1 if bernoulli else 0, _ptr(tt),
                               _ptr(pr), npairs, _ptr(out), _ptr(idx), _ptr(Z))
    if rc != 0:
        raise ValueError("oracle_decode: bad arguments")
    return (out, idx, Z) if want_Z else (out, idx)


def cdf(q, k, seq_lens, b: int, h: int, scale: float | None = None):
    """Unnormalised CDF W [n_b] fp64 and the max score m of one (b, h)."""
    qb, kb = _bits(q), _bits(k)
    B, H_q, d = qb.shape
    _, H_kv, n_max, _ = kb.shape
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(B))
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(d)))
    W = np.zeros(max(int(sl[b]), 1), dtype=np.float64)
    m = np.zeros(1, dtype=np.float64)
    rc = _load().oracle_cdf(B, H_q, H_kv, d, n_max, ctypes.c_float(scale), _ptr(qb), _ptr(kb),
                            _ptr(sl), b, h, _ptr(W), _ptr(m))
    if rc != 0:
        raise ValueError("oracle_cdf: bad arguments")
    return W[: int(sl[b])], float(m[0])


def gather(v, seq_lens, idx) -> np.ndarray:
    """(1/S) * sum_s v_{idx} in fp64 for the given indices [B,H_q,S]."""
    vb = _bits(v)
    B, H_kv, n_max, d = vb.shape
    ix = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
    _, H_q, S = ix.shape
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(B))
    out = np.zeros((B, H_q, d), dtype=np.float64)
    if _load().oracle_gather(B, H_q, H_kv, d, n_max, _ptr(vb), _ptr(sl), _ptr(ix), S, _ptr(out)) != 0:
        raise ValueError("oracle_gather: index out of range or bad arguments")
    return out
