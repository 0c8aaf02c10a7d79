"""Seeded synthetic inputs for the CSA2 step, shared by the tests, the smoke
check and the benchmark.

This module only draws numbers: it holds none of the method's arithmetic (no
quantisation, scoring, selection or attention).  Every value comes from a
counter-based 32-bit integer hash evaluated with int64 torch ops whose products
never overflow, so the same call gives bit-identical tensors on the CPU and on
a GPU.  Sub-ranges can be regenerated on their own (counters are absolute
element indices), which lets a CPU check rebuild just the rows it needs.

Value recipes (workload shapes follow the pages' decode and prefill settings):
  latent C, compression logits Z, indexer keys, indexer queries: ~N(0, 1) by an
      Irwin-Hall sum of four 16-bit uniforms (|x| < 2 sqrt 3, well inside the
      sqrt(512) latent bound); optionally RMS-scaled to norm sqrt(512);
  head weights w: U(0, 1);
  attention queries q: ~N(0, 1/512), rounded to bf16;
  window KV: ~N(0, 1), rounded to bf16;
  exact-integer mode: keys and queries integers in [-8, 8], w in multiples of
      1/16, so every fp32 product and partial sum of the indexer is exact;
  exact-compression mode (m > 1): latents on a 2^-10 grid in [-8, 8] and Z
      equal within each block, so the block average is exact in fp32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

_M32 = 0xFFFFFFFF
_SQRT3 = 1.7320508075688772


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for 0 <= x < 2^32, with no int64 overflow."""
    lo = x & 0xFFFF
    hi = x >> 16
    return (lo * c + (((hi * c) & 0xFFFF) << 16)) & _M32


def _mix32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    return x ^ (x >> 16)


def _mix32_int(x: int) -> int:
    x &= _M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & _M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & _M32
    return x ^ (x >> 16)


def hash_u32(counter: torch.Tensor, seed: int, stream: int) -> torch.Tensor:
    """32-bit hash of int64 counters (any value >= 0) under (seed, stream)."""
    key = _mix32_int(seed * 0x9E3779B1 + stream * 0x85EBCA77 + 0x165667B1)
    h = _mix32((counter & _M32) ^ key)
    return _mix32(h ^ ((counter >> 32) & _M32) ^ 0x27D4EB2F)


_CHUNK = 1 << 26


def _gen(n: int, device, fn, dtype, start: int = 0) -> torch.Tensor:
    out = torch.empty(n, dtype=dtype, device=device)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        c = torch.arange(start + s, start + e, dtype=torch.int64, device=device)
        out[s:e] = fn(c)
    return out


def uniform(shape, seed, stream, device="cpu", start=0) -> torch.Tensor:
    """U[0, 1) with 24-bit resolution, fp32."""
    n = math.prod(shape)
    f = lambda c: (hash_u32(c, seed, stream) >> 8).to(torch.float32) * (1.0 / 16777216.0)
    return _gen(n, device, f, torch.float32, start).reshape(shape)


def normal(shape, seed, stream, device="cpu", start=0) -> torch.Tensor:
    """~N(0, 1): (sum of four 16-bit uniforms - 2) * sqrt(3), fp32."""
    n = math.prod(shape)

    return _gen(n, device, lambda c: _normal_of(c, seed, stream), torch.float32,
                start).reshape(shape)


def _normal_of(c, seed, stream):
    acc = torch.zeros(c.shape, dtype=torch.float32, device=c.device)
    for i in range(4):
        u = (hash_u32(c * 4 + i, seed, stream) >> 16).to(torch.float32) * (1.0 / 65536.0)
        acc = acc + u
    return (acc - 2.0) * _SQRT3


def int_uniform(shape, lo, hi, seed, stream, device="cpu", start=0) -> torch.Tensor:
    """Integers in [lo, hi] as fp32 (exact)."""
    n = math.prod(shape)
    span = hi - lo + 1
    f = lambda c: ((hash_u32(c, seed, stream) >> 8) % span).to(torch.float32) + lo
    return _gen(n, device, f, torch.float32, start).reshape(shape)


def rms_to_sqrt512(x: torch.Tensor) -> torch.Tensor:
    """Scale each 512-vector to L2 norm sqrt(512) (the latent bound's edge)."""
    n = x.float().norm(dim=-1, keepdim=True).clamp_min(1e-30)
    return (x * (math.sqrt(512.0) / n)).to(torch.float32)


def bf16_bits(x: torch.Tensor) -> torch.Tensor:
    """Round to bf16 (RNE) and return the raw 16-bit patterns as int16."""
    return x.to(torch.bfloat16).view(torch.int16)


# ---------------------------------------------------------------- workloads
@dataclass
class Workload:
    """Sizes of one synthetic CSA2 workload (one layer call or a schedule)."""
    name: str
    batch: int               # sequences
    ctx_tokens: list         # tokens already in each sequence before the step
    new_tokens: int          # tokens appended per sequence this step (and queries)
    m: int                   # block-compression factor
    h_idx: int = 8           # indexer heads
    d_idx: int = 128         # indexer key width
    heads: int = 64          # attention query heads
    k: int = 2048            # top-k
    n_win: int = 128         # sliding window
    pool_blocks: int = 2048  # candidate-pool blocks (8 positions each)
    exact: bool = False      # exact-integer indexer inputs
    grid: bool = False       # latents on a 2^-10 grid (exact block sums)
    equal_z: bool = False    # Z equal within each block (weights exactly 1/m)
    rms_norm: bool = False   # scale latents to norm sqrt(512)
    seed: int = 1000
    sm_scale: float = 1.0
    group: int = 1           # consecutive queries sharing one sequence
    q_per_seq: int = 1       # queries per sequence (the last positions)
    extra: dict = field(default_factory=dict)


# stream ids (distinct hash streams per tensor kind)
S_C, S_Z, S_KEY, S_QIDX, S_W, S_QATT, S_WIN, S_LEN = 1, 2, 3, 4, 5, 6, 7, 8
SEQ_SHIFT = 22  # token / entry counters: (sequence << 22) + position


def latent_rows(wl: Workload, b: int, p0: int, n: int, device):
    """C and Z of tokens p0..p0+n-1 of sequence b, [n][512] fp32 each (Z is
    None when m == 1)."""
    start = ((b << SEQ_SHIFT) + p0) * 512
    if wl.grid:
        C = _gen(n * 512, device, lambda c: _grid_of(c, wl.seed), torch.float32,
                 start).reshape(n, 512)
    else:
        C = normal((n, 512), wl.seed, S_C, device, start=start)
        if wl.rms_norm:
            C = rms_to_sqrt512(C)
    Z = None
    if wl.m > 1:
        if wl.equal_z:
            Z = _gen(n * 512, device, lambda c: _equal_z(c, wl), torch.float32,
                     start).reshape(n, 512)
        else:
            Z = normal((n, 512), wl.seed, S_Z, device, start=start)
    return C, Z


def latent_rows_at(wl: Workload, b: int, entries, device="cpu"):
    """C (and Z) of the tokens of the given entries of sequence b (entry e holds
    tokens e*m .. e*m+m-1): [len(entries)][m][512] each, the same values
    latent_rows gives for those tokens."""
    e = torch.as_tensor(entries, dtype=torch.int64, device=device)
    tok = (e[:, None] * wl.m + torch.arange(wl.m, device=device)[None]).reshape(-1)
    cnt = (((b << SEQ_SHIFT) + tok) * 512)[:, None] + torch.arange(512, device=device)[None]
    if wl.grid:
        C = _grid_of(cnt, wl.seed)
    else:
        C = _normal_of(cnt, wl.seed, S_C)
        if wl.rms_norm:
            C = rms_to_sqrt512(C)
    Z = None
    if wl.m > 1:
        Z = _equal_z(cnt, wl) if wl.equal_z else _normal_of(cnt, wl.seed, S_Z)
        Z = Z.reshape(len(e), wl.m, 512)
    return C.reshape(len(e), wl.m, 512), Z


def _grid_of(cnt, seed):
    """Multiples of 2^-10 in [-8, 8]: sums of two stay exact in fp32."""
    return ((hash_u32(cnt, seed, S_C) >> 8) % 16385).to(torch.float32) * (1.0 / 1024.0) - 8.0


def _equal_z(cnt, wl):
    """Z equal over the m tokens of each entry (the weights are then exactly 1/m)."""
    tok_cnt = cnt // 512
    seq_part = tok_cnt - (tok_cnt % (1 << SEQ_SHIFT))
    ent = seq_part + (tok_cnt % (1 << SEQ_SHIFT)) // wl.m
    return _normal_of(ent * 512 + cnt % 512, wl.seed, S_Z)


def key_rows(wl: Workload, b: int, e0: int, n: int, device):
    """Indexer-key projections of entries e0..e0+n-1 of sequence b, fp32."""
    shape = (n, wl.d_idx)
    start = ((b << SEQ_SHIFT) + e0) * wl.d_idx
    if wl.exact:
        return int_uniform(shape, -8, 8, wl.seed, S_KEY, device, start=start)
    return normal(shape, wl.seed, S_KEY, device, start=start)


def query_inputs(wl: Workload, nq: int, device, layer: int = 0):
    """Indexer queries [nq][h_idx][d_idx], head weights [nq][h_idx], attention
    queries (bf16 bits) [nq][heads][512] for one layer."""
    s = wl.seed + 7919 * layer
    if wl.exact:
        qi = int_uniform((nq, wl.h_idx, wl.d_idx), -8, 8, s, S_QIDX, device)
        w = int_uniform((nq, wl.h_idx), 0, 16, s, S_W, device) * (1.0 / 16.0)
    else:
        qi = normal((nq, wl.h_idx, wl.d_idx), s, S_QIDX, device)
        w = uniform((nq, wl.h_idx), s, S_W, device)
    qa = bf16_bits(normal((nq, wl.heads, 512), s, S_QATT, device) * (1.0 / math.sqrt(512.0)))
    return qi, w, qa


def window_rows(wl: Workload, batch: int, wcap: int, device, layer: int = 0):
    """Window KV ring buffers [batch][wcap][512] bf16 bits for one layer."""
    s = wl.seed + 7919 * layer
    return bf16_bits(normal((batch, wcap, 512), s, S_WIN, device))


def loguniform_lengths(n: int, lo: int, hi: int, seed: int) -> list:
    u = uniform((n,), seed, S_LEN).double()
    return [int(round(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo)))))
            for x in u]


def config(idx: int, **over) -> Workload:
    """The five workload shapes (1-based index).  ctx_tokens = tokens already
    cached per sequence; the step appends new_tokens per sequence and issues
    q_per_seq queries at the last positions of each sequence."""
    if idx == 1:   # tiny Full-mode decode, m = 2, 4096 tokens -> 2048 entries
        wl = Workload("tiny_full_m2_ctx4096", 1, [4094], 2, 2, h_idx=4, d_idx=64, heads=16,
                      k=256, seed=1001)
    elif idx == 2:  # decoder Full-mode decode, 64K
        wl = Workload("decode_full_b32_ctx65536", 32, [65535] * 32, 1, 1, rms_norm=True,
                      seed=1002)
    elif idx == 3:  # decoder Reindex over the candidate pool, 1M
        wl = Workload("decode_reindex_b8_ctx1m", 8, [(1 << 20) - 1] * 8, 1, 1, rms_norm=True,
                      seed=1003)
    elif idx == 4:  # encoder prefill chunk, m = 2
        wl = Workload("prefill_m2_prefix262144_q4096", 1, [262144], 4096, 2, rms_norm=True,
                      seed=1004, group=32, q_per_seq=4096)
    elif idx == 5:  # 20-layer decoder schedule, mixed lengths
        lens = loguniform_lengths(64, 4096, 1 << 20, 1005)
        wl = Workload("decode_schedule20_b64_loguniform", 64, [x - 1 for x in lens], 1, 1,
                      rms_norm=True, seed=1005)
    else:
        raise ValueError(idx)
    for k_, v in over.items():
        setattr(wl, k_, v)
    return wl
