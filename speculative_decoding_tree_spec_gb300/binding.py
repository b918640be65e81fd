"""ctypes binding of the C ABI in include/spec_verify.h.

Argument marshalling only: every step of the verify path runs in the CUDA
library.  torch supplies device memory (the caching allocator) and the current
stream.  The library must have been built (``__graft_entry__.build()``); loading
fails loudly otherwise -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libspecverify.so")
_lock = threading.Lock()
_lib = None

SPEC_F32 = 0
SPEC_BF16 = 1
SPEC_FLAG_EXACT_SELECT = 1
SPEC_FLAG_TEST_STALL = 2
SPEC_FLAG_VISITED_ONLY = 4
SPEC_TREE_OK = 0
SPEC_ROW_NONFINITE = 1
SPEC_TREE_INVALID = 2
SPEC_ROW_TIMEOUT = 3
SPEC_PHASE_PREPARE = 1
SPEC_PHASE_ROWS = 2
SPEC_PHASE_WALK = 4
SPEC_PHASE_ALL = 7
SPEC_PHASE_LMHEAD = 8
SPEC_PHASE_ALL_FUSED = 15
SPEC_MAX_NODES = 4096
SPEC_MAX_VOCAB = 1 << 21
SPEC_STATIC_WORKSPACE_BYTES = 1 << 20
ERRORS = {0: "SPEC_OK", -1: "SPEC_ERR_INVALID_ARG", -2: "SPEC_ERR_UNSUPPORTED_DTYPE",
          -3: "SPEC_ERR_MISALIGNED", -4: "SPEC_ERR_WORKSPACE", -5: "SPEC_ERR_CUDA",
          -6: "SPEC_ERR_TOO_LARGE"}


class SamplingParams(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32),
                ("top_p", ctypes.c_float), ("flags", ctypes.c_uint32)]


class RowStats(ctypes.Structure):
    _fields_ = [("m", ctypes.c_float), ("status", ctypes.c_int32), ("s_f", ctypes.c_double),
                ("cut_key", ctypes.c_uint32), ("cut_idx", ctypes.c_int32),
                ("argmax", ctypes.c_int32), ("kept", ctypes.c_int32)]


class Counters(ctypes.Structure):
    _fields_ = [("dense_rows", ctypes.c_uint64), ("dense_bytes", ctypes.c_uint64),
                ("walk_bytes", ctypes.c_uint64), ("residual_passes", ctypes.c_uint64),
                ("final_draws", ctypes.c_uint64), ("fallback_rows", ctypes.c_uint64),
                ("reserved", ctypes.c_uint64 * 2)]


class SpecError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {ERRORS.get(code, code)} ({error_string(code)})")
        self.code = code


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"CUDA verify library missing at {LIB_PATH}; run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            L = ctypes.CDLL(LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
            L.spec_check_errors.argtypes = [P]
            L.spec_check_errors.restype = ctypes.c_int
            L.spec_check_build.argtypes = []
            L.spec_check_build.restype = ctypes.c_int
            L.spec_verify_workspace_size.argtypes = [i32, i32, i32, ctypes.c_int]
            L.spec_verify_workspace_size.restype = ctypes.c_size_t
            L.spec_verify_tree.argtypes = [P, P, ctypes.c_int, i32, i32, i32, i64, i64, P, P, i32,
                                           SamplingParams, u64, u64, P, P, P, P, P, P, P,
                                           ctypes.c_size_t, P]
            L.spec_verify_tree.restype = ctypes.c_int
            L.spec_verify_tree_phases.argtypes = [ctypes.c_uint32] + L.spec_verify_tree.argtypes
            L.spec_verify_tree_phases.restype = ctypes.c_int
            L.spec_verify_tree_noalloc.argtypes = L.spec_verify_tree.argtypes[:20] + [P]
            L.spec_verify_tree_noalloc.restype = ctypes.c_int
            L.spec_fused_lmhead_workspace_size.argtypes = [i32, i32, i32]
            L.spec_fused_lmhead_workspace_size.restype = ctypes.c_size_t
            L.spec_verify_tree_fused_lmhead.argtypes = [P, P, i32, P, i32, i32, i32, i64, P, P,
                                                        i32, SamplingParams, u64, u64, P, P, P,
                                                        P, P, P, P, P, ctypes.c_size_t, P]
            L.spec_verify_tree_fused_lmhead.restype = ctypes.c_int
            L.spec_verify_tree_fused_lmhead_phases.argtypes = (
                [ctypes.c_uint32] + L.spec_verify_tree_fused_lmhead.argtypes)
            L.spec_verify_tree_fused_lmhead_phases.restype = ctypes.c_int
            L.spec_commit_accepted_path.argtypes = [P, i32, i32, i32, i64, i64, i64, i64, P, P, P,
                                                    i32, P]
            L.spec_commit_accepted_path.restype = ctypes.c_int
            L.spec_verify_tree_per_request.argtypes = [
                ctypes.c_uint32, P, P, ctypes.c_int, i32, i32, i32, ctypes.c_int64, ctypes.c_int64,
                P, P, i32, P, P, P, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_uint64,
                P, P, P, P, P, P, P, ctypes.c_size_t, P]
            L.spec_verify_tree_per_request.restype = ctypes.c_int
            L.spec_draft_topk.argtypes = [P, ctypes.c_int, i32, i32, ctypes.c_int64, i32,
                                          ctypes.c_float, P, P, P, P]
            L.spec_draft_topk.restype = ctypes.c_int
            L.spec_draft_fused_workspace_size.argtypes = [i32, i32, i32]
            L.spec_draft_fused_workspace_size.restype = ctypes.c_size_t
            L.spec_draft_topk_fused_lmhead.argtypes = [P, P, i32, i32, i32, i32, ctypes.c_float,
                                                       P, ctypes.c_int64, P, P, P, P,
                                                       ctypes.c_size_t, P]
            L.spec_draft_topk_fused_lmhead.restype = ctypes.c_int
            L.spec_tree_expand_topk.argtypes = [P, P, i32, i32, i32, i32, i32, P, P]
            L.spec_tree_expand_topk.restype = ctypes.c_int
            L.spec_tree_build.argtypes = [P, P, P, P, i32, i32, i32, P, P, P, P, P, P, P]
            L.spec_tree_build.restype = ctypes.c_int
            L.spec_filter_rows.argtypes = [P, ctypes.c_int, i32, i32, i64, SamplingParams, P, P]
            L.spec_filter_rows.restype = ctypes.c_int
            L.spec_philox_words.argtypes = [u64, u64, P, P, i32, P, P]
            L.spec_philox_words.restype = ctypes.c_int
            L.spec_error_string.argtypes = [ctypes.c_int]
            L.spec_error_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


def error_string(code: int) -> str:
    return lib().spec_error_string(int(code)).decode()


def check_errors() -> list:
    """spec_check_errors: the checked build's two device error words (dense pass,
    walk), read and cleared; [0, 0] in the regular build.  Waits for the device."""
    words = (ctypes.c_uint32 * 2)()
    rc = lib().spec_check_errors(ctypes.addressof(words))
    if rc != 0:
        raise SpecError(rc, "spec_check_errors")
    return [int(words[0]), int(words[1])]


def params(temperature: float, top_k: int = 0, top_p: float = 1.0, flags: int = 0) -> SamplingParams:
    return SamplingParams(float(temperature), int(top_k), float(top_p), int(flags))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def workspace_size(B: int, N: int, V: int, dtype=torch.bfloat16) -> int:
    code = SPEC_BF16 if dtype == torch.bfloat16 else SPEC_F32
    return int(lib().spec_verify_workspace_size(B, N, V, code))


def _row_layout(t: torch.Tensor, B: int, N: int, V: int, broadcast: bool):
    """(row_pitch, batch_stride) in elements of a [B, N, V] tensor, or of an [N, V]
    tensor shared by every tree (batch_stride 0)."""
    if t.stride(-1) != 1:
        raise ValueError("logits rows must be contiguous in the vocabulary dimension")
    if broadcast:
        if tuple(t.shape) != (N, V):
            raise ValueError(f"broadcast logits must be [N, V] = [{N}, {V}]")
        return t.stride(0), 0
    if tuple(t.shape) != (B, N, V):
        raise ValueError(f"logits must be [B, N, V] = [{B}, {N}, {V}]")
    return t.stride(1), t.stride(0)


def verify_tree(p: torch.Tensor, q, draft_tokens: torch.Tensor, parent_idx: torch.Tensor,
                max_depth: int, temperature: float, top_k: int = 0, top_p: float = 1.0,
                seed: int = 0, offset: int = 0, flags: int = 0, *, batch_broadcast: bool = False,
                want_alpha: bool = True, want_counters: bool = False, workspace=None, out=None,
                stream=None, phases: int = SPEC_PHASE_ALL):
    """spec_verify_tree on device tensors.  Returns a dict of device tensors:
    accept_len [B], tokens [B, D+1], path [B, D+1], status [B], alpha [B, N] (if
    requested) and counters (a Counters struct, synchronised, if requested)."""
    B, N = draft_tokens.shape
    V = p.shape[-1]
    dev = p.device
    if draft_tokens.dtype != torch.int32 or parent_idx.dtype != torch.int32:
        raise TypeError("draft_tokens and parent_idx must be int32")
    if not (draft_tokens.is_contiguous() and parent_idx.is_contiguous()):
        raise ValueError("draft_tokens and parent_idx must be contiguous")
    dt = _dtype_code(p)
    pitch, bstride = _row_layout(p, B, N, V, batch_broadcast)
    if q is not None:
        if q.dtype != p.dtype:
            raise TypeError("p and q logits must share a dtype")
        if _row_layout(q, B, N, V, batch_broadcast) != (pitch, bstride):
            raise ValueError("p and q must share one layout")
    W = max_depth + 1
    if out is None:
        out = {
            "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
            "tokens": torch.empty((B, W), dtype=torch.int32, device=dev),
            "path": torch.empty((B, W), dtype=torch.int32, device=dev),
            "status": torch.empty(B, dtype=torch.int32, device=dev),
        }
        if want_alpha:
            out["alpha"] = torch.empty((B, N), dtype=torch.float32, device=dev)
    ws_bytes = int(lib().spec_verify_workspace_size(B, N, V, dt))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    counters = torch.zeros(8, dtype=torch.int64, device=dev) if want_counters else None
    rc = lib().spec_verify_tree_phases(
        int(phases), p.data_ptr(), None if q is None else q.data_ptr(), dt, B, N, V, pitch, bstride,
        draft_tokens.data_ptr(), parent_idx.data_ptr(), int(max_depth),
        params(temperature, top_k, top_p, flags), int(seed) & (2**64 - 1),
        int(offset) & (2**64 - 1), out["accept_len"].data_ptr(), out["tokens"].data_ptr(),
        out["path"].data_ptr(), out["alpha"].data_ptr() if "alpha" in out else None,
        out["status"].data_ptr(), None if counters is None else counters.data_ptr(),
        workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
    if rc != 0:
        raise SpecError(rc, "spec_verify_tree")
    if counters is not None:
        c = counters.cpu().numpy().view("uint64")
        out["counters"] = dict(zip(["dense_rows", "dense_bytes", "walk_bytes", "residual_passes",
                                    "final_draws", "fallback_rows"], [int(x) for x in c[:6]]))
    return out


def verify_tree_per_request(p: torch.Tensor, q: torch.Tensor, draft_tokens: torch.Tensor,
                            parent_idx: torch.Tensor, max_depth: int, temperature: torch.Tensor,
                            top_k=None, top_p=None, seed: int = 0, offset: int = 0,
                            flags: int = 0, *, want_alpha: bool = True,
                            want_counters: bool = False, workspace=None, stream=None,
                            phases: int = SPEC_PHASE_ALL):
    """spec_verify_tree_per_request: tree b verified under temperature[b], top_k[b],
    top_p[b] (device tensors [B]: float32, int32, float32; top_k / top_p may be None).
    Returns the same dict as verify_tree."""
    B, N = draft_tokens.shape
    V = p.shape[-1]
    dev = p.device
    if draft_tokens.dtype != torch.int32 or parent_idx.dtype != torch.int32:
        raise TypeError("draft_tokens and parent_idx must be int32")
    if q is None or q.dtype != p.dtype:
        raise TypeError("p and q logits must share a dtype")
    pitch, bstride = _row_layout(p, B, N, V, False)
    if _row_layout(q, B, N, V, False) != (pitch, bstride):
        raise ValueError("p and q must share one layout")
    for t, dt in ((temperature, torch.float32), (top_k, torch.int32), (top_p, torch.float32)):
        if t is not None and (t.dtype != dt or t.shape != (B,) or t.device != dev
                              or not t.is_contiguous()):
            raise TypeError("per-request arrays must be contiguous [B] tensors on the logits' device")
    W = max_depth + 1
    out = {
        "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
        "tokens": torch.empty((B, W), dtype=torch.int32, device=dev),
        "path": torch.empty((B, W), dtype=torch.int32, device=dev),
        "status": torch.empty(B, dtype=torch.int32, device=dev),
    }
    if want_alpha:
        out["alpha"] = torch.empty((B, N), dtype=torch.float32, device=dev)
    dt = _dtype_code(p)
    ws_bytes = int(lib().spec_verify_workspace_size(B, N, V, dt))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    counters = torch.zeros(8, dtype=torch.int64, device=dev) if want_counters else None
    rc = lib().spec_verify_tree_per_request(
        int(phases), p.data_ptr(), q.data_ptr(), dt, B, N, V, pitch, bstride,
        draft_tokens.data_ptr(), parent_idx.data_ptr(), int(max_depth), temperature.data_ptr(),
        None if top_k is None else top_k.data_ptr(), None if top_p is None else top_p.data_ptr(),
        int(flags), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
        out["accept_len"].data_ptr(), out["tokens"].data_ptr(), out["path"].data_ptr(),
        out["alpha"].data_ptr() if "alpha" in out else None, out["status"].data_ptr(),
        None if counters is None else counters.data_ptr(), workspace.data_ptr(),
        workspace.numel(), _stream_ptr(stream))
    if rc != 0:
        raise SpecError(rc, "spec_verify_tree_per_request")
    if counters is not None:
        c = counters.cpu().numpy().view("uint64")
        out["counters"] = dict(zip(["dense_rows", "dense_bytes", "walk_bytes", "residual_passes",
                                    "final_draws", "fallback_rows"], [int(x) for x in c[:6]]))
    return out


def verify_tree_noalloc(p: torch.Tensor, q, draft_tokens: torch.Tensor, parent_idx: torch.Tensor,
                        max_depth: int, temperature: float, top_k: int = 0, top_p: float = 1.0,
                        seed: int = 0, offset: int = 0, flags: int = 0, *,
                        batch_broadcast: bool = False, out: dict, counters=None, stream=None):
    """spec_verify_tree_noalloc on device tensors: the library's own scratch stands in
    for the workspace.  `out` holds caller-allocated device tensors accept_len [B],
    tokens [B, D+1], path [B, D+1], status [B] and optionally alpha [B, N];
    `counters` is an optional int64 device tensor of 8 entries.  This wrapper
    allocates nothing either."""
    B, N = draft_tokens.shape
    V = p.shape[-1]
    if draft_tokens.dtype != torch.int32 or parent_idx.dtype != torch.int32:
        raise TypeError("draft_tokens and parent_idx must be int32")
    if not (draft_tokens.is_contiguous() and parent_idx.is_contiguous()):
        raise ValueError("draft_tokens and parent_idx must be contiguous")
    dt = _dtype_code(p)
    pitch, bstride = _row_layout(p, B, N, V, batch_broadcast)
    if q is not None:
        if q.dtype != p.dtype:
            raise TypeError("p and q logits must share a dtype")
        if _row_layout(q, B, N, V, batch_broadcast) != (pitch, bstride):
            raise ValueError("p and q must share one layout")
    rc = lib().spec_verify_tree_noalloc(
        p.data_ptr(), None if q is None else q.data_ptr(), dt, B, N, V, pitch, bstride,
        draft_tokens.data_ptr(), parent_idx.data_ptr(), int(max_depth),
        params(temperature, top_k, top_p, flags), int(seed) & (2**64 - 1),
        int(offset) & (2**64 - 1), out["accept_len"].data_ptr(), out["tokens"].data_ptr(),
        out["path"].data_ptr(), out["alpha"].data_ptr() if "alpha" in out else None,
        out["status"].data_ptr(), None if counters is None else counters.data_ptr(),
        _stream_ptr(stream))
    if rc != 0:
        raise SpecError(rc, "spec_verify_tree_noalloc")
    return out


def verify_tree_fused_lmhead(features: torch.Tensor, weight: torch.Tensor, q,
                             draft_tokens: torch.Tensor, parent_idx: torch.Tensor, max_depth: int,
                             temperature: float, top_k: int = 0, top_p: float = 1.0,
                             seed: int = 0, offset: int = 0, flags: int = 0, *,
                             want_alpha: bool = True, want_counters: bool = False,
                             out=None, workspace=None, stream=None,
                             phases: int = SPEC_PHASE_ALL_FUSED):
    """spec_verify_tree_fused_lmhead on device tensors: features [B*N, d] and weight
    [V, d] bf16, q [B, N, V] bf16 (or None at temperature 0).  Returns the dict of
    verify_tree plus "p": the bf16 target logits [B, N, V] the call computed."""
    B, N = draft_tokens.shape
    V, d = weight.shape
    dev = weight.device
    if features.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise TypeError("features and weight must be bfloat16")
    if tuple(features.shape) != (B * N, d) or not features.is_contiguous() or \
            not weight.is_contiguous():
        raise ValueError("features must be contiguous [B*N, d] and weight contiguous [V, d]")
    if draft_tokens.dtype != torch.int32 or parent_idx.dtype != torch.int32:
        raise TypeError("draft_tokens and parent_idx must be int32")
    W = max_depth + 1
    if out is None:
        out = {
            "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
            "tokens": torch.empty((B, W), dtype=torch.int32, device=dev),
            "path": torch.empty((B, W), dtype=torch.int32, device=dev),
            "status": torch.empty(B, dtype=torch.int32, device=dev),
            # rows padded to a 16-byte aligned pitch
            "p": torch.empty((B, N, (V + 7) // 8 * 8), dtype=torch.bfloat16, device=dev)[..., :V],
        }
        if want_alpha:
            out["alpha"] = torch.empty((B, N), dtype=torch.float32, device=dev)
    pitch = out["p"].stride(1)
    if q is not None:
        if q.dtype != torch.bfloat16 or tuple(q.shape) != (B, N, V) or q.stride(1) != pitch or \
                q.stride(0) != N * pitch or q.stride(2) != 1:
            raise ValueError("q must be bf16 [B, N, V] with the row pitch of the p output")
    ws_bytes = int(lib().spec_fused_lmhead_workspace_size(B, N, V))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    counters = torch.zeros(8, dtype=torch.int64, device=dev) if want_counters else None
    rc = lib().spec_verify_tree_fused_lmhead_phases(
        int(phases), features.data_ptr(), weight.data_ptr(), d, None if q is None else q.data_ptr(), B, N, V,
        pitch, draft_tokens.data_ptr(), parent_idx.data_ptr(), int(max_depth),
        params(temperature, top_k, top_p, flags), int(seed) & (2**64 - 1),
        int(offset) & (2**64 - 1), out["p"].data_ptr(), out["accept_len"].data_ptr(),
        out["tokens"].data_ptr(), out["path"].data_ptr(),
        out["alpha"].data_ptr() if "alpha" in out else None, out["status"].data_ptr(),
        None if counters is None else counters.data_ptr(), workspace.data_ptr(),
        workspace.numel(), _stream_ptr(stream))
    if rc != 0:
        raise SpecError(rc, "spec_verify_tree_fused_lmhead")
    if counters is not None:
        c = counters.cpu().numpy().view("uint64")
        out["counters"] = dict(zip(["dense_rows", "dense_bytes", "walk_bytes", "residual_passes",
                                    "final_draws", "fallback_rows"], [int(x) for x in c[:6]]))
    return out


def commit_accepted_path(cache: torch.Tensor, prefix_len: torch.Tensor, accepted_path: torch.Tensor,
                         accept_len: torch.Tensor, stream=None) -> None:
    """spec_commit_accepted_path in place on a cache tensor [planes, B, positions, ...]
    whose trailing dimensions form one row per position (any dtype)."""
    if cache.dim() < 3:
        raise ValueError("cache must be [planes, B, positions, ...]")
    P, B, n_pos = cache.shape[:3]
    row_bytes = cache[0, 0, 0].numel() * cache.element_size()
    es = cache.element_size()
    if cache[0, 0, 0].numel() > 1 and not cache[0, 0, 0].is_contiguous():
        raise ValueError("each position's row must be contiguous")
    for t in (prefix_len, accepted_path, accept_len):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise TypeError("prefix_len, accepted_path and accept_len must be contiguous int32")
    rc = lib().spec_commit_accepted_path(
        cache.data_ptr(), B, P, n_pos, cache.stride(0) * es, cache.stride(1) * es,
        cache.stride(2) * es, row_bytes, prefix_len.data_ptr(), accepted_path.data_ptr(),
        accept_len.data_ptr(), accepted_path.shape[1], _stream_ptr(stream))
    if rc != 0:
        raise SpecError(rc, "spec_commit_accepted_path")


def draft_topk(logits: torch.Tensor, k: int, temperature: float = 1.0, stream=None) -> dict:
    """spec_draft_topk on [R, V] device rows (row pitch from the tensor's stride):
    tokens [R, k] int32, probs [R, k] float32, status [R] int32."""
    R, V = logits.shape
    if logits.stride(1) != 1:
        raise ValueError("rows must be contiguous")
    dev = logits.device
    out = {"tokens": torch.empty((R, k), dtype=torch.int32, device=dev),
           "probs": torch.empty((R, k), dtype=torch.float32, device=dev),
           "status": torch.empty(R, dtype=torch.int32, device=dev)}
    rc = lib().spec_draft_topk(logits.data_ptr(), _dtype_code(logits), R, V, logits.stride(0), k,
                               float(temperature), out["tokens"].data_ptr(),
                               out["probs"].data_ptr(), out["status"].data_ptr(),
                               _stream_ptr(stream))
    if rc != 0:
        raise SpecError(rc, "spec_draft_topk")
    return out


def draft_topk_fused_lmhead(features: torch.Tensor, weight: torch.Tensor, k: int,
                            temperature: float = 1.0, want_logits: bool = False, workspace=None,
                            stream=None) -> dict:
    """spec_draft_topk_fused_lmhead: features [R, d] and weight [V, d] bf16 (device,
    contiguous).  Returns tokens [R, k], probs [R, k], status [R] and, if asked, the
    bf16 logits [R, V] (a padded-pitch view)."""
    R, d = features.shape
    V, d2 = weight.shape
    if d2 != d or features.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise TypeError("features [R, d] and weight [V, d] must be bf16 with the same d")
    if not (features.is_contiguous() and weight.is_contiguous()):
        raise ValueError("features and weight must be contiguous")
    dev = features.device
    out = {"tokens": torch.empty((R, k), dtype=torch.int32, device=dev),
           "probs": torch.empty((R, k), dtype=torch.float32, device=dev),
           "status": torch.empty(R, dtype=torch.int32, device=dev)}
    logits, pitch = None, 0
    if want_logits:
        pitch = (V + 7) // 8 * 8  # rows on 16-byte boundaries
        logits = torch.empty((R, pitch), dtype=torch.bfloat16, device=dev)[:, :V]
        out["logits"] = logits
    ws_bytes = int(lib().spec_draft_fused_workspace_size(R, V, k))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    rc = lib().spec_draft_topk_fused_lmhead(
        features.data_ptr(), weight.data_ptr(), d, R, V, k, float(temperature),
        None if logits is None else logits.data_ptr(), pitch, out["tokens"].data_ptr(),
        out["probs"].data_ptr(), out["status"].data_ptr(), workspace.data_ptr(),
        workspace.numel(), _stream_ptr(stream))
    if rc != 0:
        raise SpecError(rc, "spec_draft_topk_fused_lmhead")
    return out


def tree_expand_topk(cand_parent: torch.Tensor, cand_prob: torch.Tensor, layer_begin: int,
                     layer_end: int, k: int, stream=None) -> torch.Tensor:
    """spec_tree_expand_topk: [B, k] int32 candidate numbers to expand next."""
    B, n = cand_parent.shape
    out = torch.empty((B, k), dtype=torch.int32, device=cand_parent.device)
    rc = lib().spec_tree_expand_topk(cand_parent.data_ptr(), cand_prob.data_ptr(), B, n,
                                     layer_begin, layer_end, k, out.data_ptr(), _stream_ptr(stream))
    if rc != 0:
        raise SpecError(rc, "spec_tree_expand_topk")
    return out


def tree_build(cand_parent: torch.Tensor, cand_token: torch.Tensor, cand_prob: torch.Tensor,
               root_token: torch.Tensor, m: int, stream=None) -> dict:
    """spec_tree_build: the flattened draft (tokens, parent_idx, position_ids, src, mask,
    status) of every tree."""
    B, n = cand_parent.shape
    dev = cand_parent.device
    for t in (cand_parent, cand_token, root_token):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise TypeError("candidate parents, tokens and roots must be contiguous int32")
    if cand_prob.dtype != torch.float32 or not cand_prob.is_contiguous():
        raise TypeError("cand_prob must be contiguous float32")
    M = m + 1
    out = {k: torch.empty((B, M), dtype=torch.int32, device=dev)
           for k in ("tokens", "parent_idx", "position_ids", "src")}
    out["mask"] = torch.empty((B, M, M), dtype=torch.uint8, device=dev)
    out["status"] = torch.empty(B, dtype=torch.int32, device=dev)
    rc = lib().spec_tree_build(cand_parent.data_ptr(), cand_token.data_ptr(), cand_prob.data_ptr(),
                               root_token.data_ptr(), B, n, m, out["tokens"].data_ptr(),
                               out["parent_idx"].data_ptr(), out["position_ids"].data_ptr(),
                               out["src"].data_ptr(), out["mask"].data_ptr(),
                               out["status"].data_ptr(), _stream_ptr(stream))
    if rc != 0:
        raise SpecError(rc, "spec_tree_build")
    return out


def verify_tree_host(p_host: torch.Tensor, q_host, tokens_host: torch.Tensor,
                     parents_host: torch.Tensor, max_depth: int, temperature: float,
                     top_k: int = 0, top_p: float = 1.0, seed: int = 0, offset: int = 0,
                     device="cuda", staging=None, stream=None):
    """End-to-end call on host (ideally pinned) tensors: copies the inputs to the
    device, verifies, and copies accept_len / tokens / path back.  `staging` may
    hold preallocated device buffers (keys p, q, tokens, parents, workspace, out)."""
    st = staging if staging is not None else {}
    def dev_like(name, t):
        if name not in st:
            st[name] = torch.empty(t.shape, dtype=t.dtype, device=device)
        st[name].copy_(t, non_blocking=True)
        return st[name]
    p = dev_like("p", p_host)
    q = None if q_host is None else dev_like("q", q_host)
    tok = dev_like("tokens", tokens_host)
    par = dev_like("parents", parents_host)
    res = verify_tree(p, q, tok, par, max_depth, temperature, top_k, top_p, seed, offset,
                      want_alpha=False, workspace=st.get("workspace"), out=st.get("out"),
                      stream=stream)
    st.setdefault("out", res)
    host = {k: res[k].to("cpu", non_blocking=True) for k in ("accept_len", "tokens", "path")}
    torch.cuda.current_stream().synchronize()
    return host


def filter_rows(logits: torch.Tensor, temperature: float, top_k: int = 0, top_p: float = 1.0,
                flags: int = 0, stream=None):
    """spec_filter_rows on a [R, V] device tensor.  Returns a dict of device tensors
    m, status, s_f, cut_key (int64), cut_idx, argmax, kept."""
    if logits.dim() != 2 or logits.stride(-1) != 1:
        raise ValueError("logits must be [R, V] with contiguous rows")
    R, V = logits.shape
    stats = torch.empty((max(R, 1), 32), dtype=torch.uint8, device=logits.device)
    rc = lib().spec_filter_rows(logits.data_ptr(), _dtype_code(logits), R, V, logits.stride(0),
                                params(temperature, top_k, top_p, flags), stats.data_ptr(),
                                _stream_ptr(stream))
    if rc != 0:
        raise SpecError(rc, "spec_filter_rows")
    stats = stats[:R]
    i32 = stats.view(torch.int32)
    return {
        "m": stats.view(torch.float32)[:, 0],
        "status": i32[:, 1],
        "s_f": stats.view(torch.float64)[:, 1],
        "cut_key": i32[:, 4].to(torch.int64) & 0xFFFFFFFF,
        "cut_idx": i32[:, 5],
        "argmax": i32[:, 6],
        "kept": i32[:, 7],
    }


def philox_words(seed: int, offset: int, b_idx: torch.Tensor, node_idx: torch.Tensor, stream=None):
    """[n, 4] int64 tensor of the Philox words for (seed, offset, b_idx[i], node_idx[i])."""
    n = b_idx.numel()
    out = torch.empty((max(n, 1), 4), dtype=torch.int32, device=b_idx.device)
    rc = lib().spec_philox_words(int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                 b_idx.data_ptr(), node_idx.data_ptr(), n, out.data_ptr(),
                                 _stream_ptr(stream))
    if rc != 0:
        raise SpecError(rc, "spec_philox_words")
    return out[:n].to(torch.int64) & 0xFFFFFFFF


class PreparedVerify:
    """A spec_verify_tree_phases call with every argument fixed (device tensors
    allocated once), for loops that call the same verify step many times."""

    def __init__(self, p, q, draft_tokens, parent_idx, max_depth, temperature, top_k=0,
                 top_p=1.0, seed=0, offset=0, flags=0, batch_broadcast=False, stream=None,
                 per_request=None):
        """per_request: optional (temperature [B] f32, top_k [B] i32 or None, top_p [B]
        f32 or None) device tensors -- spec_verify_tree_per_request then replaces the
        scalar temperature / top_k / top_p."""
        B, N = draft_tokens.shape
        V = p.shape[-1]
        dev = p.device
        dt = _dtype_code(p)
        pitch, bstride = _row_layout(p, B, N, V, batch_broadcast)
        if q is not None and _row_layout(q, B, N, V, batch_broadcast) != (pitch, bstride):
            raise ValueError("p and q must share one layout")
        W = max_depth + 1
        self.out = {
            "accept_len": torch.empty(B, dtype=torch.int32, device=dev),
            "tokens": torch.empty((B, W), dtype=torch.int32, device=dev),
            "path": torch.empty((B, W), dtype=torch.int32, device=dev),
            "status": torch.empty(B, dtype=torch.int32, device=dev),
        }
        self.counters = torch.zeros(8, dtype=torch.int64, device=dev)
        ws_bytes = int(lib().spec_verify_workspace_size(B, N, V, dt))
        self.workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
        self._keep = (p, q, draft_tokens, parent_idx, per_request)
        if per_request is not None:
            T_r, k_r, p_r = per_request
            self._fn = lib().spec_verify_tree_per_request
            self._args = [
                p.data_ptr(), q.data_ptr(), dt, B, N, V, pitch, bstride, draft_tokens.data_ptr(),
                parent_idx.data_ptr(), int(max_depth), T_r.data_ptr(),
                None if k_r is None else k_r.data_ptr(), None if p_r is None else p_r.data_ptr(),
                int(flags), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                self.out["accept_len"].data_ptr(), self.out["tokens"].data_ptr(),
                self.out["path"].data_ptr(), None, self.out["status"].data_ptr(), None,
                self.workspace.data_ptr(), self.workspace.numel(), _stream_ptr(stream)]
            self._counter_args = list(self._args)
            self._counter_args[22] = self.counters.data_ptr()
            return
        self._fn = lib().spec_verify_tree_phases
        self._args = [
            p.data_ptr(), None if q is None else q.data_ptr(), dt, B, N, V, pitch, bstride,
            draft_tokens.data_ptr(), parent_idx.data_ptr(), int(max_depth),
            params(temperature, top_k, top_p, flags), int(seed) & (2**64 - 1),
            int(offset) & (2**64 - 1), self.out["accept_len"].data_ptr(),
            self.out["tokens"].data_ptr(), self.out["path"].data_ptr(), None,
            self.out["status"].data_ptr(), None, self.workspace.data_ptr(),
            self.workspace.numel(), _stream_ptr(stream)]
        self._counter_args = list(self._args)
        self._counter_args[19] = self.counters.data_ptr()

    def __call__(self, phases: int = SPEC_PHASE_ALL) -> None:
        rc = self._fn(phases, *self._args)
        if rc != 0:
            raise SpecError(rc, "spec_verify_tree_phases")

    def read_counters(self) -> dict:
        """Run the whole step once more with the work counters requested; returns them."""
        rc = self._fn(SPEC_PHASE_ALL, *self._counter_args)
        if rc != 0:
            raise SpecError(rc, "spec_verify_tree_phases")
        c = self.counters.cpu().numpy().view("uint64")
        return dict(zip(["dense_rows", "dense_bytes", "walk_bytes", "residual_passes",
                         "final_draws", "fallback_rows"], [int(x) for x in c[:6]]))
