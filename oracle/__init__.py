"""CPU oracle for batched tree speculative-sampling verification.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The product library
never imports this package, and this package never imports the product.

The arithmetic lives in ``spec_oracle.c`` (plain C, fp64); this module only
compiles it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libspec_oracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1
NEAR = 1e-6


class RowInfo(ctypes.Structure):
    _fields_ = [
        ("status", ctypes.c_int32),
        ("argmax", ctypes.c_int32),
        ("kept", ctypes.c_int32),
        ("cut_idx", ctypes.c_int32),
        ("m", ctypes.c_double),
        ("cut_z", ctypes.c_double),
        ("s_k", ctypes.c_double),
        ("s_f", ctypes.c_double),
        ("near", ctypes.c_int32),
        ("pad", ctypes.c_int32),
        ("margin", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libspec_oracle.so`` (gcc, -O2)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # SPEC_ORACLE_LIB points the pins at another build of this file (the
            # mutation test plants mistakes in a copy to show the pins catch them).
            lib = ctypes.CDLL(os.environ.get("SPEC_ORACLE_LIB") or build())
            P = ctypes.c_void_p
            lib.oracle_philox4x32_10.argtypes = [P, P, P]
            lib.oracle_philox4x32_10.restype = None
            lib.oracle_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.c_int]
            lib.oracle_uniform.restype = ctypes.c_double
            lib.oracle_uniform_from_word.argtypes = [ctypes.c_uint32]
            lib.oracle_uniform_from_word.restype = ctypes.c_double
            lib.oracle_filter_row.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                              ctypes.c_int, ctypes.c_double, P, P]
            lib.oracle_filter_row.restype = ctypes.c_int
            lib.oracle_filter_rows.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                               ctypes.c_double, P, P]
            lib.oracle_filter_rows.restype = None
            lib.oracle_verify_tree.argtypes = [
                P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int64, ctypes.c_int64, P, P, ctypes.c_int, ctypes.c_double,
                ctypes.c_int, ctypes.c_double, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int32,
                P, P,
                P, P, P, P, P, P, P, ctypes.c_int]
            lib.oracle_verify_tree.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _as_logits(x):
    """Return (contiguous array, dtype code).  bf16 logits are passed as raw uint16 bits."""
    x = np.asarray(x)
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), F32
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), BF16
    raise TypeError(f"oracle logits must be float32 or raw bf16 bits (uint16), got {x.dtype}")


def philox4x32_10(ctr, key):
    """Philox4x32-10 of a 4-word counter under a 2-word key -> 4 uint32 words."""
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, offset: int, b: int, node: int, word: int) -> float:
    return _load().oracle_uniform(seed, offset, b, node, word)


def uniform_from_word(x: int) -> float:
    return _load().oracle_uniform_from_word(x)


def filter_row(row, temperature: float, top_k: int, top_p: float, want_probs: bool = True):
    """Filter one logit row.  Returns (probs or None, RowInfo)."""
    r, dt = _as_logits(row)
    V = r.shape[-1]
    probs = np.zeros(V, dtype=np.float64) if want_probs else None
    info = RowInfo()
    _load().oracle_filter_row(_ptr(r), dt, V, float(temperature), int(top_k), float(top_p),
                              _ptr(probs), ctypes.byref(info))
    return probs, info


def filter_rows(rows, temperature: float, top_k: int, top_p: float, want_probs: bool = False):
    """Filter every row of a [R, V] array.  Returns (probs [R, V] or None, list of RowInfo)."""
    r, dt = _as_logits(rows)
    R, V = r.shape
    infos = (RowInfo * R)()
    probs = np.zeros((R, V), dtype=np.float64) if want_probs else None
    _load().oracle_filter_rows(_ptr(r), dt, R, V, V, float(temperature), int(top_k),
                               float(top_p), _ptr(probs), infos)
    return probs, list(infos)


NEAR_BITS = {"p_cut": 1, "q_cut": 2, "accept": 4, "draw": 8}


def near_reasons(bits: int):
    """Names of the near-boundary decisions in one tree's near bits."""
    return [k for k, v in NEAR_BITS.items() if int(bits) & v]


def verify_tree(logits_p, logits_q, draft_tokens, parent_idx, max_depth: int,
                temperature: float, top_k: int, top_p: float, seed: int, offset: int = 0,
                u_accept=None, u_final=None, want_final_dist: bool = False,
                batch_broadcast: bool = False, nthreads: int = 1, batch_index: int = 0):
    """Run the oracle walk on B trees.

    logits_p / logits_q: [B, N, V] (or [N, V] with batch_broadcast=True, shared by
    every tree) float32 or raw-bf16 uint16.  draft_tokens / parent_idx: [B, N] int32.
    Tree b draws its uniforms as batch index batch_index + b.
    Returns a dict of numpy arrays: accept_len [B], tokens [B, D+1], path [B, D+1],
    alpha [B, N], status [B], near [B] and optionally final_dist [B, V].
    near[b] marks the decisions of tree b that fell within 1e-6 of their boundary,
    where rounding order alone could flip them: bit NEAR_BITS["p_cut"] (a p row's
    top-p cut), "q_cut", "accept" (|r - alpha|) and "draw" (the final inverse CDF).
    """
    p, dt = _as_logits(logits_p)
    q, dq = _as_logits(logits_q)
    if dt != dq:
        raise TypeError("p and q logits must share a dtype")
    tokens = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    parent = np.ascontiguousarray(parent_idx, dtype=np.int32)
    B, N = tokens.shape
    V = p.shape[-1]
    if batch_broadcast:
        if p.shape != (N, V) or q.shape != (N, V):
            raise ValueError("broadcast logits must be [N, V]")
        batch_stride = 0
    else:
        if p.shape != (B, N, V) or q.shape != (B, N, V):
            raise ValueError("logits must be [B, N, V]")
        batch_stride = N * V
    W = max_depth + 1
    out = {
        "accept_len": np.zeros(B, dtype=np.int32),
        "tokens": np.zeros((B, W), dtype=np.int32),
        "path": np.zeros((B, W), dtype=np.int32),
        "alpha": np.zeros((B, N), dtype=np.float64),
        "status": np.zeros(B, dtype=np.int32),
        "near": np.zeros(B, dtype=np.int32),
    }
    if want_final_dist:
        out["final_dist"] = np.zeros((B, V), dtype=np.float64)
    ua = None if u_accept is None else np.ascontiguousarray(u_accept, dtype=np.float64)
    uf = None if u_final is None else np.ascontiguousarray(u_final, dtype=np.float64)
    if ua is not None and ua.shape != (B, N):
        raise ValueError("u_accept must be [B, N]")
    if uf is not None and uf.shape != (B, N):
        raise ValueError("u_final must be [B, N]")
    _load().oracle_verify_tree(
        _ptr(p), _ptr(q), dt, B, N, V, V, batch_stride, _ptr(tokens), _ptr(parent),
        int(max_depth), float(temperature), int(top_k), float(top_p), int(seed) & (2**64 - 1),
        int(offset) & (2**64 - 1), int(batch_index), _ptr(ua), _ptr(uf), _ptr(out["accept_len"]),
        _ptr(out["tokens"]), _ptr(out["path"]), _ptr(out["alpha"]), _ptr(out["status"]),
        _ptr(out["near"]), _ptr(out.get("final_dist")), int(nthreads))
    return out


def verify_tree_per_request(logits_p, logits_q, draft_tokens, parent_idx, max_depth: int,
                            temperature, top_k, top_p, seed: int, offset: int = 0):
    """Per-request sampling parameters (one batch serving requests with different
    settings).  Reading taken here: tree b is verified exactly as a batch of one under
    its own temperature[b], top_k[b], top_p[b], drawing its uniforms as batch index b;
    a tree whose values are invalid (temperature negative or not finite, top_p <= 0 or
    NaN, top_k < 0) gets status 2 (invalid) and accept_len -1."""
    tokens = np.asarray(draft_tokens)
    B = tokens.shape[0]
    outs = []
    for b in range(B):
        T, k, p = float(temperature[b]), int(top_k[b]), float(top_p[b])
        if not (np.isfinite(T) and T >= 0.0) or not (p > 0.0) or k < 0:
            outs.append(None)
            continue
        outs.append(verify_tree(logits_p[b:b + 1], logits_q[b:b + 1], tokens[b:b + 1],
                                np.asarray(parent_idx)[b:b + 1], max_depth, T, k, p, seed,
                                offset, batch_index=b))
    return outs

