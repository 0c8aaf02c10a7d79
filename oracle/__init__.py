"""Float64 CPU oracle for the CSA2 global-attention step (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never does: it shares no code with this oracle.

The arithmetic lives in ``csa2_oracle.c`` (plain C, float64, bit-level FP4/FP8);
this module compiles it with gcc and wraps it with numpy arrays.  Parity pins
for every function are in ``tests/test_oracle_pins.py``.  Functions with no pin
other than the oracle itself: none of the arithmetic; absolute attention and
score values at random inputs are pinned only through the special cases
(dense attention via a library routine, ReLU-GEMV, exact-integer scoring).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa2_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libcsa2_oracle.so")
_lock = threading.Lock()
_lib = None

FULL, REINDEX, REUSE = 0, 1, 2
D = 512


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, -O2, OpenMP when available). Returns the .so path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The compiled oracle.  CSA2_ORACLE_LIB, when set, names another build of
    this source to load instead (the mutation test loads copies with a
    planted mistake that way)."""
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("CSA2_ORACLE_LIB") or build()
            L = ctypes.CDLL(path)
            dbl, i32, i64, vp = ctypes.c_double, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
            L.or_e2m1_value.restype = dbl
            L.or_e2m1_value.argtypes = [i32]
            L.or_e4m3_value.restype = dbl
            L.or_e4m3_value.argtypes = [i32]
            L.or_e4m3_nearest.restype = i32
            L.or_e4m3_nearest.argtypes = [dbl]
            L.or_fp8_pow2_scale.restype = dbl
            L.or_fp8_pow2_scale.argtypes = [dbl]
            L.or_fp4_scale_byte.restype = i32
            L.or_fp4_scale_byte.argtypes = [dbl, vp]
            L.or_fp4_code.restype = i32
            L.or_fp4_code.argtypes = [dbl, dbl]
            L.or_fp4_encode_entry.restype = i32
            L.or_fp4_encode_entry.argtypes = [vp, vp, vp]
            L.or_fp4_decode_entry.restype = None
            L.or_fp4_decode_entry.argtypes = [vp, vp, vp]
            L.or_fp8_encode_rows.restype = None
            L.or_fp8_encode_rows.argtypes = [vp, i64, i32, vp, vp]
            L.or_compress_block.restype = None
            L.or_compress_block.argtypes = [vp, vp, i32, vp]
            L.or_append.restype = i64
            L.or_append.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
            L.or_append_project.restype = i64
            L.or_append_project.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
            L.or_scores_full.restype = None
            L.or_scores_full.argtypes = [vp, vp, i32, i32, vp, vp, i64, i64, vp]
            L.or_scores_at.restype = None
            L.or_scores_at.argtypes = [vp, vp, i32, i32, vp, vp, vp, i64, vp]
            L.or_topk.restype = i32
            L.or_topk.argtypes = [vp, vp, i64, i32, vp]
            L.or_topk_f32.restype = i32
            L.or_topk_f32.argtypes = [vp, vp, i64, i32, vp]
            L.or_pool.restype = i32
            L.or_pool.argtypes = [vp, i64, i32, vp, vp]
            L.or_blockmax.restype = None
            L.or_blockmax.argtypes = [vp, i64, vp]
            L.or_gather_rows.restype = i32
            L.or_gather_rows.argtypes = [vp, vp, i64, vp, i32, vp, i32, i64, i64, i32, vp]
            L.or_attention.restype = None
            L.or_attention.argtypes = [i32, vp, i64, vp, dbl, vp, vp]
            L.or_layer.restype = None
            L.or_layer.argtypes = [i32, vp, vp, vp, i32, vp, vp, vp, vp]
            L.or_max_threads.restype = i32
            L.or_set_threads.argtypes = [i32]
            _lib = L
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- formats
def e2m1_value(nib: int) -> float:
    return lib().or_e2m1_value(int(nib))


def e4m3_value(b: int) -> float:
    return lib().or_e4m3_value(int(b))


def e4m3_nearest(y: float) -> int:
    return lib().or_e4m3_nearest(float(y))


def fp8_pow2_scale(amax: float) -> float:
    return lib().or_fp8_pow2_scale(float(amax))


def fp4_scale_byte(amax: float):
    sat = ctypes.c_int(0)
    b = lib().or_fp4_scale_byte(float(amax), ctypes.byref(sat))
    return b, sat.value


def fp4_code(x: float, s: float) -> int:
    return lib().or_fp4_code(float(x), float(s))


def fp4_encode_entry(x):
    x = _c(x, np.float64)
    assert x.shape == (D,)
    codes = np.zeros(D // 2, np.uint8)
    scales = np.zeros(D // 16, np.uint8)
    nsat = lib().or_fp4_encode_entry(_p(x), _p(codes), _p(scales))
    return codes, scales, nsat


def fp4_decode_entry(codes, scales):
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    out = np.zeros(D, np.float64)
    lib().or_fp4_decode_entry(_p(codes), _p(scales), _p(out))
    return out


def fp4_decode_rows(codes, scales):
    """Dequantise rows: codes [n][256], scales [n][32] -> float64 [n][512]."""
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    n = codes.shape[0]
    out = np.zeros((n, D), np.float64)
    for r in range(n):
        lib().or_fp4_decode_entry(_p(codes[r]), _p(scales[r]), _p(out[r]))
    return out


def fp8_encode_rows(x):
    x = _c(x, np.float32)
    rows, d = x.reshape(-1, x.shape[-1]).shape
    out = np.zeros((rows, d), np.uint8)
    sc = np.zeros(rows, np.float32)
    lib().or_fp8_encode_rows(_p(x), rows, d, _p(out), _p(sc))
    return out.reshape(x.shape), sc.reshape(x.shape[:-1])


def e4m3_values(b):
    """Vectorised decode of E4M3 bytes via the oracle's scalar decoder."""
    table = np.array([e4m3_value(i) for i in range(256)], np.float64)
    return table[np.asarray(b, np.int64)]


def compress_block(C, Z, m):
    C = _c(C, np.float32).reshape(m, D)
    Zp = None if m == 1 else _c(Z, np.float32).reshape(m, D)
    out = np.zeros(D, np.float64)
    lib().or_compress_block(_p(C), _p(Zp), m, _p(out))
    return out


def append(C, Z, key, m):
    """C, Z: [B][n_tok][512] fp32, key: [B][n_tok/m][d_idx] fp32.
    Returns codes [B*ne][256], scales [B*ne][32], kidx [B*ne][d_idx],
    kscale [B*ne] fp32, the fp64 compressed latents [B*ne][512], and the
    number of saturated groups."""
    C = _c(C, np.float32)
    B, n_tok, _ = C.shape
    Zc = _c(Z, np.float32) if m > 1 else None
    key = _c(key, np.float32)
    d_idx = key.shape[-1]
    ne = n_tok // m
    codes = np.zeros((B * ne, D // 2), np.uint8)
    scales = np.zeros((B * ne, D // 16), np.uint8)
    kidx = np.zeros((B * ne, d_idx), np.uint8)
    ksc = np.zeros(B * ne, np.float32)
    x = np.zeros((B * ne, D), np.float64)
    nsat = lib().or_append(B, n_tok, m, d_idx, _p(C), _p(Zc), _p(key), _p(codes), _p(scales),
                           _p(kidx), _p(ksc), _p(x))
    return codes, scales, kidx, ksc, x, int(nsat)


def append_project(C, Z, w_ik, m):
    """Append whose indexer key is the dequantised entry times W_IK.
    C, Z: [B][n_tok][512] fp32; w_ik: [512][d_idx] bf16 bit patterns (uint16).
    Returns codes, scales, kidx, kscale as append() does, the fp64 keys before
    FP8 encoding [B*ne][d_idx], and the number of saturated groups."""
    C = _c(C, np.float32)
    B, n_tok, _ = C.shape
    Zc = _c(Z, np.float32) if m > 1 else None
    w_ik = _c(w_ik, np.uint16)
    d_idx = w_ik.shape[1]
    ne = n_tok // m
    codes = np.zeros((B * ne, D // 2), np.uint8)
    scales = np.zeros((B * ne, D // 16), np.uint8)
    kidx = np.zeros((B * ne, d_idx), np.uint8)
    ksc = np.zeros(B * ne, np.float32)
    k = np.zeros((B * ne, d_idx), np.float64)
    nsat = lib().or_append_project(B, n_tok, m, d_idx, _p(C), _p(Zc), _p(w_ik), _p(codes),
                                   _p(scales), _p(kidx), _p(ksc), _p(k))
    return codes, scales, kidx, ksc, k, int(nsat)


# ----------------------------------------------------------------- indexer
def scores_full(kidx, kscale, q, w, base, n):
    """Full-mode scores of one query (q [h_idx][d_idx] fp32, w [h_idx]) over
    cache rows base..base+n-1."""
    kidx, kscale = _c(kidx, np.uint8), _c(kscale, np.float32)
    q, w = _c(q, np.float32), _c(w, np.float32)
    h_idx, d_idx = q.shape
    out = np.zeros(max(n, 1), np.float64)
    lib().or_scores_full(_p(kidx), _p(kscale), d_idx, h_idx, _p(q), _p(w), int(base), int(n), _p(out))
    return out[:n]


def scores_at(kidx, kscale, q, w, rows):
    kidx, kscale = _c(kidx, np.uint8), _c(kscale, np.float32)
    q, w = _c(q, np.float32), _c(w, np.float32)
    rows = _c(rows, np.int64)
    h_idx, d_idx = q.shape
    out = np.zeros(max(len(rows), 1), np.float64)
    lib().or_scores_at(_p(kidx), _p(kscale), d_idx, h_idx, _p(q), _p(w), _p(rows), len(rows), _p(out))
    return out[: len(rows)]


def topk(scores, k, pos=None):
    """Positions of the k largest scores (ties -> lower position), ascending."""
    if np.asarray(scores).dtype == np.float32:
        s = _c(scores, np.float32)
        fn = lib().or_topk_f32
    else:
        s = _c(scores, np.float64)
        fn = lib().or_topk
    pp = None if pos is None else _c(pos, np.int32)
    out = np.zeros(max(min(k, len(s)), 1), np.int32)
    cnt = fn(_p(s), _p(pp), len(s), int(k), _p(out))
    return out[:cnt]


def blockmax(scores):
    s = _c(scores, np.float64)
    out = np.zeros(max((len(s) + 7) // 8, 1), np.float64)
    lib().or_blockmax(_p(s), len(s), _p(out))
    return out[: (len(s) + 7) // 8]


def pool(scores, nblk_max=2048):
    """Returns (ascending block ids, number of visible positions)."""
    s = _c(scores, np.float64)
    blk = np.zeros(max(nblk_max, 1), np.int32)
    nb = ctypes.c_int(0)
    pn = lib().or_pool(_p(s), len(s), int(nblk_max), _p(blk), ctypes.byref(nb))
    return blk[: nb.value], int(pn)


# ----------------------------------------------------------------- attention
def gather_rows(codes, scales, seq_base, idx, win, wcap, t, s, n_win):
    """win: [wcap][512] uint16 (bf16 bits) of this query's sequence or None."""
    codes, scales = _c(codes, np.uint8), _c(scales, np.uint8)
    idx = _c(idx, np.int32)
    wv = None if win is None else _c(win, np.uint16)
    rows = np.zeros((len(idx) + n_win + 1, D), np.float64)
    n = lib().or_gather_rows(_p(codes), _p(scales), int(seq_base), _p(idx), len(idx), _p(wv),
                             int(wcap), int(t), int(s), int(n_win), _p(rows))
    return rows[:n]


def attention(q_bf16_bits, rows, sm_scale):
    """q: [H][512] uint16 bf16 bits; rows: [n][512] float64."""
    q = _c(q_bf16_bits, np.uint16)
    rows = _c(rows, np.float64)
    H = q.shape[0]
    out = np.zeros((H, D), np.float64)
    lse = np.zeros(H, np.float64)
    lib().or_attention(H, _p(q), rows.shape[0], _p(rows), float(sm_scale), _p(out), _p(lse))
    return out, lse


# ----------------------------------------------------------------- layer
class _LayerArgs(ctypes.Structure):
    _fields_ = [
        ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("kidx", ctypes.c_void_p),
        ("kscale", ctypes.c_void_p), ("seq_base", ctypes.c_void_p),
        ("d_idx", ctypes.c_int), ("m", ctypes.c_int),
        ("nq", ctypes.c_int), ("q_seq", ctypes.c_void_p), ("q_pos", ctypes.c_void_p),
        ("h_idx", ctypes.c_int), ("q_idx", ctypes.c_void_p), ("w", ctypes.c_void_p),
        ("k", ctypes.c_int), ("pool_blocks", ctypes.c_int),
        ("H", ctypes.c_int), ("q_attn", ctypes.c_void_p), ("win", ctypes.c_void_p),
        ("wcap", ctypes.c_int), ("n_win", ctypes.c_int), ("win_start", ctypes.c_void_p),
        ("sm_scale", ctypes.c_double),
    ]


def layer(mode, *, codes, scales, kidx, kscale, seq_base, m, q_seq, q_pos, k, H, q_attn,
          win, wcap, n_win, sm_scale, q_idx=None, w=None, win_start=None, idx=None, cnt=None,
          pool_blk=None, pool_n=None, build_pool=False, pool_blocks=2048):
    """One CSA2 layer for a batch of queries, in float64.

    Returns dict(idx [nq][k], cnt [nq], out [nq][H][512], lse [nq][H],
    pool_blk, pool_n)."""
    keep = []

    def arr(a, dt):
        if a is None:
            return None
        a = _c(a, dt)
        keep.append(a)
        return a

    codes, scales = arr(codes, np.uint8), arr(scales, np.uint8)
    kidx = arr(kidx, np.uint8) if kidx is not None else None
    kscale = arr(kscale, np.float32) if kscale is not None else None
    seq_base = arr(seq_base, np.int64)
    q_seq, q_pos = arr(q_seq, np.int32), arr(q_pos, np.int32)
    nq = len(q_seq)
    q_idx = arr(q_idx, np.float32)
    w = arr(w, np.float32)
    h_idx = q_idx.shape[1] if q_idx is not None else 0
    d_idx = kidx.shape[1] if kidx is not None else 0
    q_attn = arr(q_attn, np.uint16)
    win = arr(win, np.uint16)
    win_start = arr(win_start, np.int32)
    a = _LayerArgs(_p(codes), _p(scales), _p(kidx), _p(kscale), _p(seq_base), d_idx, m, nq,
                   _p(q_seq), _p(q_pos), h_idx, _p(q_idx), _p(w), k, pool_blocks, H, _p(q_attn),
                   _p(win), wcap, n_win, _p(win_start), float(sm_scale))
    idx_io = np.zeros((nq, k), np.int32) if idx is None else np.array(idx, np.int32, copy=True)
    cnt_io = np.zeros(nq, np.int32) if cnt is None else np.array(cnt, np.int32, copy=True)
    if pool_blk is None:
        pool_blk = np.zeros((nq, pool_blocks), np.int32)
        pool_n = np.zeros(nq, np.int32)
    else:
        pool_blk = np.array(pool_blk, np.int32, copy=True)
        pool_n = np.array(pool_n, np.int32, copy=True)
    out = np.zeros((nq, H, D), np.float64)
    lse = np.zeros((nq, H), np.float64)
    lib().or_layer(int(mode), ctypes.byref(a), _p(idx_io), _p(cnt_io), int(build_pool),
                   _p(pool_blk), _p(pool_n), _p(out), _p(lse))
    return dict(idx=idx_io, cnt=cnt_io, out=out, lse=lse, pool_blk=pool_blk, pool_n=pool_n)


def max_threads() -> int:
    return lib().or_max_threads()


def set_threads(n: int) -> None:
    lib().or_set_threads(int(n))
