"""Thin Python binding of the CSA2 C ABI (include/csa2.h).

Argument marshalling only: tensors become device pointers, and every step of
the path runs in the CUDA library libcsa2.so.  There is no fallback: if the
library is missing or a call fails, an exception is raised.  PyTorch supplies
device memory and the current CUDA stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

FULL, REINDEX, REUSE = 0, 1, 2
D = 512
CNT_FP4_SATURATED, CNT_CAPACITY, CNT_BAD_INPUT, CNT_TIMEOUT = 0, 1, 2, 3
NUM_COUNTERS = 4

_lock = threading.Lock()
_lib = None

_STATUS = {0: "ok", -1: "invalid argument", -2: "pointer not 16-byte aligned",
           -3: "workspace or output too small", -4: "shape not supported", -5: "CUDA error"}

EXPORTS = ["csa2_quantize_append", "csa2_quantize_append_project", "csa2_index_full", "csa2_index_reindex", "csa2_topk",
           "csa2_pool_select", "csa2_sparse_attn", "csa2_layer_step", "csa2_index_workspace_size",
           "csa2_topk_workspace_size", "csa2_attn_workspace_size", "csa2_layer_workspace_size",
           "csa2_status_string", "csa2_launch_count", "csa2_topk_noalloc",
           "csa2_topk_noalloc_max_scratch"]


class CsaError(RuntimeError):
    pass


class _Cache(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("kidx", ctypes.c_void_p),
                ("kscale", ctypes.c_void_p), ("seq_base", ctypes.c_void_p),
                ("seq_len", ctypes.c_void_p), ("cap", ctypes.c_int64), ("batch", ctypes.c_int32),
                ("d_idx", ctypes.c_int32), ("m", ctypes.c_int32)]


class _Queries(ctypes.Structure):
    _fields_ = [("q_seq", ctypes.c_void_p), ("q_pos", ctypes.c_void_p), ("nq", ctypes.c_int32),
                ("group", ctypes.c_int32)]


class _LayerArgs(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("cache", ctypes.c_void_p), ("queries", ctypes.c_void_p),
                ("q_idx", ctypes.c_void_p), ("w", ctypes.c_void_p), ("h_idx", ctypes.c_int32),
                ("max_n", ctypes.c_int64), ("k", ctypes.c_int32), ("build_pool", ctypes.c_int32),
                ("pool_blocks", ctypes.c_int32), ("pool_blk", ctypes.c_void_p),
                ("pool_n", ctypes.c_void_p), ("idx", ctypes.c_void_p), ("cnt", ctypes.c_void_p),
                ("q", ctypes.c_void_p), ("H", ctypes.c_int32), ("win", ctypes.c_void_p),
                ("wcap", ctypes.c_int32), ("win_start", ctypes.c_void_p),
                ("n_win", ctypes.c_int32), ("sm_scale", ctypes.c_float), ("out", ctypes.c_void_p),
                ("lse", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("ws_bytes", ctypes.c_size_t), ("counters", ctypes.c_void_p)]


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """Loads libcsa2.so, building it with nvcc first if it is missing or stale."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            if not os.path.exists(path):
                raise CsaError(f"CUDA library not found at {path}")
            L = ctypes.CDLL(path)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            sig = {
                "csa2_quantize_append": [vp, vp, vp, vp, i32, vp, vp],
                "csa2_quantize_append_project": [vp, vp, vp, vp, i32, vp, vp],
                "csa2_index_full": [vp, vp, vp, vp, i32, i64, vp, i64, vp, i64, vp, vp, sz, vp, vp],
                "csa2_index_reindex": [vp, vp, vp, vp, i32, vp, vp, i32, vp, i64, vp, vp, sz, vp,
                                       vp],
                "csa2_topk": [vp, i64, vp, vp, i32, i32, i64, i32, vp, i64, vp, vp, sz, vp],
                "csa2_pool_select": [vp, i64, vp, i32, i64, i32, vp, vp, vp, sz, vp],
                "csa2_sparse_attn": [vp, vp, vp, i64, vp, i32, vp, i32, vp, i32, vp, i32,
                                     ctypes.c_float, vp, vp, vp, sz, vp, vp],
                "csa2_layer_step": [vp, vp],
            }
            for name, args in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = ctypes.c_int
            L.csa2_index_workspace_size.argtypes = [i32, i32, i32, i32]
            L.csa2_index_workspace_size.restype = sz
            L.csa2_topk_workspace_size.argtypes = [i32, i64]
            L.csa2_topk_workspace_size.restype = sz
            L.csa2_attn_workspace_size.argtypes = [i32, i32, i32, i32]
            L.csa2_attn_workspace_size.restype = sz
            L.csa2_layer_workspace_size.argtypes = [vp]
            L.csa2_layer_workspace_size.restype = sz
            L.csa2_status_string.argtypes = [ctypes.c_int]
            L.csa2_status_string.restype = ctypes.c_char_p
            L.csa2_launch_count.argtypes = []
            L.csa2_launch_count.restype = ctypes.c_uint64
            _lib = L
    return _lib


def _check(status: int, what: str):
    if status != 0:
        raise CsaError(f"{what}: {_STATUS.get(status, status)}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise CsaError("tensor is not on a CUDA device")
    if not t.is_contiguous():
        raise CsaError("tensor is not contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def launch_count() -> int:
    return int(lib().csa2_launch_count())


# ---------------------------------------------------------------- state
class Cache:
    """An FP4 main-KV cache with FP8 indexer keys, in device memory.

    `lengths_cap[b]` is the capacity of sequence b (entries); rows are laid
    out back to back with each sequence starting on a multiple of 8."""

    def __init__(self, lengths_cap, d_idx: int, m: int, device="cuda"):
        caps = [int(-(-int(c) // 8) * 8) for c in lengths_cap]
        base = [0]
        for c in caps:
            base.append(base[-1] + c)
        self.batch = len(caps)
        self.cap = max(8, base[-1])
        self.d_idx = d_idx
        self.m = m
        dev = torch.device(device)
        self.codes = torch.zeros(self.cap, 256, dtype=torch.uint8, device=dev)
        self.scales = torch.zeros(self.cap, 32, dtype=torch.uint8, device=dev)
        self.kidx = torch.zeros(self.cap, d_idx, dtype=torch.uint8, device=dev)
        self.kscale = torch.zeros(self.cap, dtype=torch.float32, device=dev)
        self.seq_base = torch.tensor(base, dtype=torch.int64, device=dev)
        self.seq_len = torch.zeros(self.batch, dtype=torch.int32, device=dev)
        self.base_host = base

    def struct(self, seq=None) -> _Cache:
        """The C struct; with seq = b, a one-sequence view of sequence b."""
        if seq is None:
            return _Cache(self.codes.data_ptr(), self.scales.data_ptr(), self.kidx.data_ptr(),
                          self.kscale.data_ptr(), self.seq_base.data_ptr(), self.seq_len.data_ptr(),
                          self.cap, self.batch, self.d_idx, self.m)
        return _Cache(self.codes.data_ptr(), self.scales.data_ptr(), self.kidx.data_ptr(),
                      self.kscale.data_ptr(), self.seq_base.data_ptr() + 8 * int(seq),
                      self.seq_len.data_ptr() + 4 * int(seq), self.cap, 1, self.d_idx, self.m)


class Queries:
    def __init__(self, q_seq, q_pos, group: int = 1, device="cuda"):
        self.q_seq = torch.as_tensor(q_seq, dtype=torch.int32).to(device).contiguous()
        self.q_pos = torch.as_tensor(q_pos, dtype=torch.int32).to(device).contiguous()
        self.nq = int(self.q_seq.numel())
        self.group = group

    def struct(self) -> _Queries:
        return _Queries(self.q_seq.data_ptr(), self.q_pos.data_ptr(), self.nq, self.group)


def new_counters(device="cuda"):
    return torch.zeros(NUM_COUNTERS, dtype=torch.int32, device=device)


def workspace(nbytes: int, device="cuda"):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- entry points
def quantize_append(cache: Cache, C, Z, key, counters=None, seq=None):
    """Appends C.shape[1] tokens to every sequence (or only to sequence `seq`)."""
    n_tok = int(C.shape[1])
    cs = cache.struct(seq)
    _check(lib().csa2_quantize_append(ctypes.byref(cs), _ptr(C), _ptr(Z), _ptr(key), n_tok,
                                      _ptr(counters), _stream()), "csa2_quantize_append")


def quantize_append_project(cache: Cache, C, Z, w_ik, counters=None, seq=None):
    """Appends C.shape[1] tokens to every sequence (or only to sequence `seq`),
    each entry's indexer key projected from the stored entry by w_ik, a bf16
    tensor [512][d_idx]."""
    if w_ik.dtype != torch.bfloat16 or tuple(w_ik.shape) != (512, cache.d_idx):
        raise CsaError(f"w_ik must be bf16 [512][{cache.d_idx}], got {w_ik.dtype} {tuple(w_ik.shape)}")
    n_tok = int(C.shape[1])
    cs = cache.struct(seq)
    _check(lib().csa2_quantize_append_project(ctypes.byref(cs), _ptr(C), _ptr(Z),
                                              _ptr(w_ik.contiguous()), n_tok, _ptr(counters),
                                              _stream()),
           "csa2_quantize_append_project")


def index_workspace_size(nq, group, h_idx, d_idx) -> int:
    return int(lib().csa2_index_workspace_size(nq, group, h_idx, d_idx))


def topk_workspace_size(nq, max_n) -> int:
    return int(lib().csa2_topk_workspace_size(nq, max_n))


def attn_workspace_size(nq, H, k_max, n_win) -> int:
    return int(lib().csa2_attn_workspace_size(nq, H, k_max, n_win))


def index_full(cache: Cache, qs: Queries, q_idx, w, max_n, scores, blockmax=None, n_valid=None,
               ws=None, counters=None):
    h_idx = int(q_idx.shape[1])
    if ws is None:
        ws = workspace(index_workspace_size(qs.nq, qs.group, h_idx, cache.d_idx), q_idx.device)
    cs, qq = cache.struct(), qs.struct()
    _check(lib().csa2_index_full(ctypes.byref(cs), ctypes.byref(qq), _ptr(q_idx), _ptr(w), h_idx,
                                 int(max_n), _ptr(scores), int(scores.shape[1]), _ptr(blockmax),
                                 int(blockmax.shape[1]) if blockmax is not None else 0,
                                 _ptr(n_valid), _ptr(ws), ws.numel(), _ptr(counters), _stream()),
           "csa2_index_full")


def index_reindex(cache: Cache, qs: Queries, q_idx, w, pool_blk, pool_n, scores, n_valid=None,
                  ws=None, counters=None):
    h_idx = int(q_idx.shape[1])
    if ws is None:
        ws = workspace(index_workspace_size(qs.nq, 1, h_idx, cache.d_idx), q_idx.device)
    cs, qq = cache.struct(), qs.struct()
    _check(lib().csa2_index_reindex(ctypes.byref(cs), ctypes.byref(qq), _ptr(q_idx), _ptr(w),
                                    h_idx, _ptr(pool_blk), _ptr(pool_n), int(pool_blk.shape[1]),
                                    _ptr(scores), int(scores.shape[1]), _ptr(n_valid), _ptr(ws),
                                    ws.numel(), _ptr(counters), _stream()), "csa2_index_reindex")


def topk(scores, n_valid, k, idx_out, cnt_out, max_n=None, pool_blk=None, ws=None):
    nq = int(scores.shape[0])
    max_n = int(scores.shape[1] if max_n is None else max_n)
    if ws is None:
        ws = workspace(topk_workspace_size(nq, max_n), scores.device)
    _check(lib().csa2_topk(_ptr(scores), int(scores.shape[1]), _ptr(n_valid), _ptr(pool_blk),
                           int(pool_blk.shape[1]) if pool_blk is not None else 0, nq, max_n,
                           int(k), _ptr(idx_out), int(idx_out.shape[1]), _ptr(cnt_out), _ptr(ws),
                           ws.numel(), _stream()), "csa2_topk")


def pool_select(blockmax, n_valid, max_n, pool_blk, pool_n, ws=None):
    nq = int(blockmax.shape[0])
    if ws is None:
        ws = workspace(topk_workspace_size(nq, (int(max_n) + 7) // 8), blockmax.device)
    _check(lib().csa2_pool_select(_ptr(blockmax), int(blockmax.shape[1]), _ptr(n_valid), nq,
                                  int(max_n), int(pool_blk.shape[1]), _ptr(pool_blk),
                                  _ptr(pool_n), _ptr(ws), ws.numel(), _stream()),
           "csa2_pool_select")


def sparse_attn(cache: Cache, qs: Queries, idx, cnt, q, win, n_win, out, lse=None, win_start=None,
                sm_scale=1.0, k_max=None, ws=None, counters=None):
    H = int(q.shape[1])
    k_max = int(idx.shape[1] if (k_max is None and idx is not None) else (k_max or 0))
    wcap = int(win.shape[1]) if win is not None else 0
    if ws is None:
        ws = workspace(attn_workspace_size(qs.nq, H, k_max, n_win), q.device)
    cs, qq = cache.struct(), qs.struct()
    _check(lib().csa2_sparse_attn(ctypes.byref(cs), ctypes.byref(qq), _ptr(idx),
                                  int(idx.shape[1]) if idx is not None else 0, _ptr(cnt), k_max,
                                  _ptr(q), H, _ptr(win), wcap, _ptr(win_start), int(n_win),
                                  float(sm_scale), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(),
                                  _ptr(counters), _stream()), "csa2_sparse_attn")


class Layer:
    """Arguments of one csa2_layer_step call; keeps the ctypes structures alive."""

    def __init__(self, mode, cache: Cache, qs: Queries, *, k, q, win, n_win, out, idx, cnt,
                 q_idx=None, w=None, max_n=0, build_pool=False, pool_blocks=2048, pool_blk=None,
                 pool_n=None, lse=None, win_start=None, sm_scale=1.0, counters=None, ws=None):
        self._cs = cache.struct()
        self._qs = qs.struct()
        self._keep = [q_idx, w, pool_blk, pool_n, idx, cnt, q, win, win_start, out, lse, counters]
        a = _LayerArgs()
        a.mode = int(mode)
        a.cache = ctypes.addressof(self._cs)
        a.queries = ctypes.addressof(self._qs)
        a.q_idx = q_idx.data_ptr() if q_idx is not None else None
        a.w = w.data_ptr() if w is not None else None
        a.h_idx = int(q_idx.shape[1]) if q_idx is not None else 0
        a.max_n = int(max_n)
        a.k = int(k)
        a.build_pool = int(bool(build_pool))
        a.pool_blocks = int(pool_blocks)
        a.pool_blk = pool_blk.data_ptr() if pool_blk is not None else None
        a.pool_n = pool_n.data_ptr() if pool_n is not None else None
        a.idx = idx.data_ptr()
        a.cnt = cnt.data_ptr()
        a.q = q.data_ptr()
        a.H = int(q.shape[1])
        a.win = win.data_ptr() if win is not None else None
        a.wcap = int(win.shape[1]) if win is not None else 0
        a.win_start = win_start.data_ptr() if win_start is not None else None
        a.n_win = int(n_win)
        a.sm_scale = float(sm_scale)
        a.out = out.data_ptr()
        a.lse = lse.data_ptr() if lse is not None else None
        a.counters = counters.data_ptr() if counters is not None else None
        self.args = a
        need = int(lib().csa2_layer_workspace_size(ctypes.byref(a)))
        if ws is None or ws.numel() < need:
            ws = workspace(need, q.device)
        self.ws = ws
        a.workspace = ws.data_ptr()
        a.ws_bytes = ws.numel()

    def __call__(self):
        _check(lib().csa2_layer_step(ctypes.byref(self.args), _stream()), "csa2_layer_step")
