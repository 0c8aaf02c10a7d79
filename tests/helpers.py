"""Shared test plumbing: builds a workload's cache on the GPU (through the C ABI)
and the matching rows on the CPU (through the oracle), from the same seeded
generator.  No expected value here comes from the CUDA path."""
import numpy as np
import pytest
import torch

import csa2_inputs as ci
import oracle as O
import sparse_attention_decode_step_gb300 as csa

TOL = 2e-3   # max |gpu - oracle| / max |oracle| per row (scores, attention outputs)


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def bits16(t):
    """bf16 tensor bits (int16 torch) -> numpy uint16."""
    return t.detach().cpu().numpy().view(np.uint16)


def rel_rows(g, r):
    g = np.asarray(g, np.float64).reshape(-1, np.asarray(g).shape[-1])
    r = np.asarray(r, np.float64).reshape(g.shape)
    den = np.maximum(np.abs(r).max(1), 1e-30)
    return (np.abs(g - r).max(1) / den)


def append_seq(cache, wl, b, n_tok, device, chunk=32768, counters=None):
    """Appends tokens seq_len*m .. +n_tok of sequence b through the GPU append."""
    done = 0
    start_tok = int(cache.seq_len[b].item()) * wl.m
    while done < n_tok:
        n = min(chunk, n_tok - done)
        n -= n % wl.m
        C, Z = ci.latent_rows(wl, b, start_tok + done, n, device)
        key = ci.key_rows(wl, b, (start_tok + done) // wl.m, n // wl.m, device)
        csa.quantize_append(cache, C[None].contiguous(), None if Z is None else Z[None].contiguous(),
                            key[None].contiguous(), counters=counters, seq=b)
        done += n


def build_gpu_cache(wl, device="cuda", extra_entries=8, counters=None):
    caps = [(t + wl.new_tokens) // wl.m + extra_entries for t in wl.ctx_tokens]
    cache = csa.Cache(caps, wl.d_idx, wl.m, device)
    for b, t in enumerate(wl.ctx_tokens):
        if t:
            append_seq(cache, wl, b, t, device, counters=counters)
    return cache


def oracle_rows(wl, b, e0, n):
    """Oracle-encoded entries e0..e0+n-1 of sequence b: codes, scales, kidx, kscale, x."""
    C, Z = ci.latent_rows(wl, b, e0 * wl.m, n * wl.m, "cpu")
    key = ci.key_rows(wl, b, e0, n, "cpu")
    codes, scales, kidx, ksc, x, _ = O.append(C.numpy()[None], None if Z is None else Z.numpy()[None],
                                              key.numpy()[None], wl.m)
    return codes, scales, kidx, ksc, x


def oracle_seq_cache(wl, b, n):
    """The first n entries of sequence b, oracle-encoded, as a one-sequence cache."""
    codes, scales, kidx, ksc, _ = oracle_rows(wl, b, 0, n)
    return dict(codes=codes, scales=scales, kidx=kidx, kscale=ksc, seq_base=[0])
