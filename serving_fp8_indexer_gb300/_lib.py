"""ctypes binding of libsmla (include/smla.h).

Argument marshalling only: every function checks that the torch tensors it
is handed have the dtype, device and layout the C ABI expects, passes their
device pointers and the current CUDA stream, and raises SmlaError when the
library returns a non-OK status.  There is no fallback: if libsmla.so is
missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsmla.so")

SMLA_OK = 0
STATUS_NAMES = {0: "SMLA_OK", 1: "SMLA_ERR_INVALID_ARG", 2: "SMLA_ERR_UNSUPPORTED", 3: "SMLA_ERR_CUDA",
                4: "SMLA_ERR_TIMEOUT", 5: "SMLA_ERR_DEVICE_CHECK"}
SMLA_BF16 = 0
SMLA_E4M3 = 1

EXPORTED = ("smla_indexer_scores", "smla_topk_workspace_size", "smla_topk", "smla_indexer_topk_workspace_size",
            "smla_indexer_topk", "smla_sparse_prefill",
            "smla_sparse_prefill_bf16_cache", "smla_dense_prefill", "smla_sparse_decode_workspace_size", "smla_sparse_decode",
            "smla_sparse_decode_noalloc",
            "smla_check_device_errors", "smla_selftest_wait_timeout", "smla_last_error", "smla_version")


class SmlaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class SeqsT(ctypes.Structure):
    _fields_ = [("cu_q", ctypes.c_void_p), ("kv_len", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("B", ctypes.c_int32), ("max_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("T", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads libsmla.so (built by serving_fp8_indexer_gb300.build) and declares
    the C signatures.  Raises OSError if the library is absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise OSError(f"libsmla.so not found at {p}; build it with serving_fp8_indexer_gb300.build")
        lib = ctypes.CDLL(p)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        lib.smla_indexer_scores.argtypes = [vp, vp, vp, vp, i64, SeqsT, i32, vp, i64, vp]
        sz = ctypes.c_size_t
        lib.smla_topk_workspace_size.argtypes = [i32, i64, i32]
        lib.smla_topk_workspace_size.restype = sz
        lib.smla_topk.argtypes = [vp, i64, SeqsT, i32, vp, vp, vp, sz, vp]
        lib.smla_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
        lib.smla_indexer_topk_workspace_size.argtypes = [i32, i64, i32, i32]
        lib.smla_indexer_topk_workspace_size.restype = sz
        lib.smla_indexer_topk.argtypes = [vp, vp, vp, vp, i64, SeqsT, i32, i64, i32, vp, vp, vp, sz, vp]
        lib.smla_sparse_prefill_bf16_cache.argtypes = [vp, vp, i64, vp, i32, vp, i32, i32, i32, f32, vp, vp, vp]
        lib.smla_dense_prefill.argtypes = [vp, i32, vp, i64, vp, i32, SeqsT, i32, i32, f32, vp, vp, vp]
        lib.smla_sparse_decode_workspace_size.argtypes = [i32, i32, i32]
        lib.smla_sparse_decode_workspace_size.restype = sz
        lib.smla_sparse_decode.argtypes = [vp, i32, vp, i64, vp, i32, vp, i32, vp, i32, i32, i32, f32, vp, vp, vp,
                                           sz, vp]
        lib.smla_sparse_decode_noalloc.argtypes = [vp, i32, vp, i64, vp, i32, vp, i32, vp, i32, i32, i32, f32, vp,
                                                   vp, vp]
        lib.smla_sparse_prefill.argtypes = [vp, i32, vp, i64, vp, i32, vp, i32, vp, i32, i32, i32, f32, vp, vp, vp]
        lib.smla_check_device_errors.argtypes = [vp]
        lib.smla_last_error.argtypes = [ctypes.c_char_p, ctypes.c_size_t]
        lib.smla_last_error.restype = ctypes.c_size_t
        lib.smla_version.restype = ctypes.c_char_p
        for name in ("smla_indexer_scores", "smla_topk", "smla_indexer_topk", "smla_sparse_prefill",
                     "smla_sparse_prefill_bf16_cache",
                     "smla_dense_prefill",
                     "smla_sparse_decode", "smla_sparse_decode_noalloc", "smla_check_device_errors",
                     "smla_selftest_wait_timeout"):
            getattr(lib, name).restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def last_error(lib=None) -> str:
    lib = lib or load()
    buf = ctypes.create_string_buffer(1024)
    lib.smla_last_error(buf, len(buf))
    return buf.value.decode(errors="replace")


def _check(lib, status: int):
    if status != SMLA_OK:
        raise SmlaError(status, last_error(lib))


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor], dtype, name: str, ndim: Optional[int] = None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    return t.data_ptr() if t.numel() else None


class Seqs:
    """Device-side ragged batch over a paged cache (see smla_seqs_t)."""

    def __init__(self, cu_q: torch.Tensor, kv_len: torch.Tensor, page_table: torch.Tensor, page_size: int, T: int):
        self.cu_q, self.kv_len, self.page_table = cu_q, kv_len, page_table
        self.page_size, self.T = int(page_size), int(T)
        self.B = int(kv_len.shape[0])
        self.max_pages = int(page_table.shape[1])

    @classmethod
    def from_host(cls, seqs, device="cuda"):
        """From the generator's host-side Seqs (numpy arrays)."""
        return cls(torch.from_numpy(seqs.cu_q).to(device), torch.from_numpy(seqs.kv_len).to(device),
                   torch.from_numpy(seqs.page_table).to(device), seqs.page_size, seqs.T)

    def as_c(self) -> SeqsT:
        return SeqsT(_ptr(self.cu_q, torch.int32, "cu_q", 1), _ptr(self.kv_len, torch.int32, "kv_len", 1),
                     _ptr(self.page_table, torch.int32, "page_table", 2), self.B, self.max_pages, self.page_size,
                     self.T)


def indexer_scores(q: torch.Tensor, q_scale: torch.Tensor, k_pool: torch.Tensor, k_scale: torch.Tensor,
                   seqs: Seqs, scores: torch.Tensor, stream=None) -> torch.Tensor:
    """scores[t, key] for every key of t's sequence (-inf past pos(t)).
    q uint8 e4m3 [T, H_idx, 128]; q_scale f32 [T, H_idx]; k_pool uint8 e4m3
    [phys_rows, 128]; k_scale f32 [phys_rows]; scores f32 [T, score_stride]."""
    lib = load()
    T, H_idx = (int(q.shape[0]), int(q.shape[1])) if q.dim() == 3 else (0, 0)
    st = lib.smla_indexer_scores(_ptr(q, torch.uint8, "q", 3), _ptr(q_scale, torch.float32, "q_scale", 2),
                                 _ptr(k_pool, torch.uint8, "k_pool", 2), _ptr(k_scale, torch.float32, "k_scale", 1),
                                 int(k_pool.shape[0]), seqs.as_c(), H_idx,
                                 _ptr(scores, torch.float32, "scores", 2), int(scores.shape[1]), _stream(stream))
    _check(lib, st)
    if T != seqs.T:
        raise ValueError("q.shape[0] != seqs.T")
    return scores


def topk_workspace_size(T: int, score_stride: int, k: int) -> int:
    """Bytes of device scratch smla_topk needs for these sizes."""
    return int(load().smla_topk_workspace_size(int(T), int(score_stride), int(k)))


def topk(scores: torch.Tensor, seqs: Seqs, k: int, indices: torch.Tensor, topk_lengths: torch.Tensor,
         workspace: Optional[torch.Tensor] = None, stream=None):
    """indices uint32 [T, k] physical rows (tail 0xFFFFFFFF), topk_lengths uint32 [T].
    workspace: a uint8 CUDA tensor of at least topk_workspace_size() bytes,
    or None when that size is 0."""
    lib = load()
    ws = _ptr(workspace, torch.uint8, "workspace") if workspace is not None else None
    wsb = int(workspace.numel()) if workspace is not None else 0
    st = lib.smla_topk(_ptr(scores, torch.float32, "scores", 2), int(scores.shape[1]), seqs.as_c(), int(k),
                       _ptr(indices, torch.uint32, "indices", 2), _ptr(topk_lengths, torch.uint32, "topk_lengths", 1),
                       ws, wsb, _stream(stream))
    _check(lib, st)
    return indices, topk_lengths


def indexer_topk_workspace_size(T: int, score_stride: int, H_idx: int, k: int) -> int:
    """Bytes of device scratch smla_indexer_topk needs (0 when rows stay on chip)."""
    return int(load().smla_indexer_topk_workspace_size(int(T), int(score_stride), int(H_idx), int(k)))


def indexer_topk(q: torch.Tensor, q_scale: torch.Tensor, k_pool: torch.Tensor, k_scale: torch.Tensor, seqs: Seqs,
                 score_stride: int, k: int, indices: torch.Tensor, topk_lengths: torch.Tensor,
                 workspace: Optional[torch.Tensor] = None, stream=None):
    """Fused indexer + top-k: indices uint32 [T, k] and topk_lengths uint32 [T]
    as indexer_scores followed by topk, without the score buffer (rows of up
    to 128 * H_idx keys; longer ones use `workspace`)."""
    lib = load()
    H_idx = int(q.shape[1]) if q.dim() == 3 else 0
    ws = _ptr(workspace, torch.uint8, "workspace") if workspace is not None else None
    wsb = int(workspace.numel()) if workspace is not None else 0
    st = lib.smla_indexer_topk(_ptr(q, torch.uint8, "q", 3), _ptr(q_scale, torch.float32, "q_scale", 2),
                               _ptr(k_pool, torch.uint8, "k_pool", 2), _ptr(k_scale, torch.float32, "k_scale", 1),
                               int(k_pool.shape[0]), seqs.as_c(), H_idx, int(score_stride), int(k),
                               _ptr(indices, torch.uint32, "indices", 2),
                               _ptr(topk_lengths, torch.uint32, "topk_lengths", 1), ws, wsb, _stream(stream))
    _check(lib, st)
    return indices, topk_lengths


def _q_arg(q: torch.Tensor):
    if q.dtype == torch.bfloat16:
        return SMLA_BF16, _ptr(q, torch.bfloat16, "q", 3)
    return SMLA_E4M3, _ptr(q, torch.uint8, "q", 3)


def sparse_prefill(q: torch.Tensor, latent: torch.Tensor, scales: Optional[torch.Tensor], scale_block_size: int,
                   indices: torch.Tensor, topk_lengths: torch.Tensor, softmax_scale: float, out: torch.Tensor,
                   attn_sink: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out bf16 [T, H, 512] = sparse MLA prefill.  q is bf16 or uint8 (e4m3
    bytes) [T, H, 576]; latent uint8 e4m3 [phys_rows, 576]; scales f32
    [phys_rows, ceil(576/sbs)] or None; indices uint32 [T, stride];
    topk_lengths uint32 [T]; attn_sink f32 [H] or None."""
    lib = load()
    qd, qp = _q_arg(q)
    T, H = int(q.shape[0]), int(q.shape[1])
    st = lib.smla_sparse_prefill(qp, qd, _ptr(latent, torch.uint8, "latent", 2), int(latent.shape[0]),
                                 _ptr(scales, torch.float32, "scales", 2), int(scale_block_size),
                                 _ptr(indices, torch.uint32, "indices", 2), int(indices.shape[1]),
                                 _ptr(topk_lengths, torch.uint32, "topk_lengths", 1), T, H, int(out.shape[2]),
                                 float(softmax_scale), _ptr(attn_sink, torch.float32, "attn_sink", 1),
                                 _ptr(out, torch.bfloat16, "out", 3), _stream(stream))
    _check(lib, st)
    return out


def sparse_prefill_bf16_cache(q: torch.Tensor, latent: torch.Tensor, indices: torch.Tensor,
                              topk_lengths: torch.Tensor, softmax_scale: float, out: torch.Tensor,
                              attn_sink: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Sparse MLA prefill over a BF16 latent cache: q bf16 [T, H, 576], latent
    bf16 [phys_rows, 576]; the other arguments as sparse_prefill."""
    lib = load()
    T, H = int(q.shape[0]), int(q.shape[1])
    st = lib.smla_sparse_prefill_bf16_cache(_ptr(q, torch.bfloat16, "q", 3), _ptr(latent, torch.bfloat16, "latent", 2),
                                            int(latent.shape[0]), _ptr(indices, torch.uint32, "indices", 2),
                                            int(indices.shape[1]), _ptr(topk_lengths, torch.uint32, "topk_lengths", 1),
                                            T, H, int(out.shape[2]), float(softmax_scale),
                                            _ptr(attn_sink, torch.float32, "attn_sink", 1),
                                            _ptr(out, torch.bfloat16, "out", 3), _stream(stream))
    _check(lib, st)
    return out


def dense_prefill(q: torch.Tensor, latent: torch.Tensor, scales: Optional[torch.Tensor], scale_block_size: int,
                  seqs: Seqs, softmax_scale: float, out: torch.Tensor, attn_sink: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """out bf16 [T, H, 512] = dense causal MLA prefill: every token attends to
    every key 0..pos of its sequence through the page table."""
    lib = load()
    qd, qp = _q_arg(q)
    if int(q.shape[0]) != seqs.T:
        raise ValueError("q.shape[0] != seqs.T")
    st = lib.smla_dense_prefill(qp, qd, _ptr(latent, torch.uint8, "latent", 2), int(latent.shape[0]),
                                _ptr(scales, torch.float32, "scales", 2), int(scale_block_size), seqs.as_c(),
                                int(q.shape[1]), int(out.shape[2]), float(softmax_scale),
                                _ptr(attn_sink, torch.float32, "attn_sink", 1), _ptr(out, torch.bfloat16, "out", 3),
                                _stream(stream))
    _check(lib, st)
    return out


def sparse_decode_workspace_size(T: int, H: int, indices_stride: int) -> int:
    """Bytes of device scratch smla_sparse_decode needs on the current device."""
    return int(load().smla_sparse_decode_workspace_size(int(T), int(H), int(indices_stride)))


def sparse_decode(q: torch.Tensor, latent: torch.Tensor, scales: Optional[torch.Tensor], scale_block_size: int,
                  indices: torch.Tensor, topk_lengths: torch.Tensor, softmax_scale: float, out: torch.Tensor,
                  workspace: Optional[torch.Tensor], attn_sink: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """Sparse MLA decode (split-K over each token's keys); the arguments of
    sparse_prefill plus a uint8 CUDA workspace of at least
    sparse_decode_workspace_size() bytes (None when that is 0)."""
    lib = load()
    qd, qp = _q_arg(q)
    T, H = int(q.shape[0]), int(q.shape[1])
    ws = _ptr(workspace, torch.uint8, "workspace") if workspace is not None else None
    wsb = int(workspace.numel()) if workspace is not None else 0
    st = lib.smla_sparse_decode(qp, qd, _ptr(latent, torch.uint8, "latent", 2), int(latent.shape[0]),
                                _ptr(scales, torch.float32, "scales", 2), int(scale_block_size),
                                _ptr(indices, torch.uint32, "indices", 2), int(indices.shape[1]),
                                _ptr(topk_lengths, torch.uint32, "topk_lengths", 1), T, H, int(out.shape[2]),
                                float(softmax_scale), _ptr(attn_sink, torch.float32, "attn_sink", 1),
                                _ptr(out, torch.bfloat16, "out", 3), ws, wsb, _stream(stream))
    _check(lib, st)
    return out


def sparse_decode_noalloc(q: torch.Tensor, latent: torch.Tensor, scales: Optional[torch.Tensor],
                          scale_block_size: int, indices: torch.Tensor, topk_lengths: torch.Tensor,
                          softmax_scale: float, out: torch.Tensor, attn_sink: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """sparse_decode for callers that cannot allocate device memory: no
    workspace argument; the split partials use the library's fixed device
    scratch (see smla_sparse_decode_noalloc in include/smla.h)."""
    lib = load()
    qd, qp = _q_arg(q)
    T, H = int(q.shape[0]), int(q.shape[1])
    st = lib.smla_sparse_decode_noalloc(qp, qd, _ptr(latent, torch.uint8, "latent", 2), int(latent.shape[0]),
                                        _ptr(scales, torch.float32, "scales", 2), int(scale_block_size),
                                        _ptr(indices, torch.uint32, "indices", 2), int(indices.shape[1]),
                                        _ptr(topk_lengths, torch.uint32, "topk_lengths", 1), T, H,
                                        int(out.shape[2]), float(softmax_scale),
                                        _ptr(attn_sink, torch.float32, "attn_sink", 1),
                                        _ptr(out, torch.bfloat16, "out", 3), _stream(stream))
    _check(lib, st)
    return out


def check_device_errors(stream=None):
    lib = load()
    _check(lib, lib.smla_check_device_errors(_stream(stream)))


def selftest_wait_timeout(limit_us: int, stream=None):
    """Enqueues the device timeout self-test (see smla_selftest_wait_timeout)."""
    lib = load()
    _check(lib, lib.smla_selftest_wait_timeout(int(limit_us), _stream(stream)))


def version() -> str:
    return load().smla_version().decode()
