"""Full-size workloads through the public layer call, checked on sampled
queries that the oracle recomputes one by one.

Indexer inputs are in exact-integer mode (every score exact in fp32 and
float64), so top-k lists and candidate pools must match the oracle exactly;
attention outputs are compared within 2e-3 of the row's max |oracle| value.
Inputs are drawn on the GPU by the seeded generator and copied to the host for
the oracle (the generator gives identical values on both devices)."""
import numpy as np
import pytest
import torch

import csa2_inputs as ci
import oracle as O
import sparse_attention_decode_step_gb300 as csa
from helpers import TOL, bits16, need_gpu, rel_rows
from sparse_attention_decode_step_gb300 import schedule as S

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"


@pytest.fixture(autouse=True)
def _gpu():
    need_gpu()


def _np(t):
    return t.detach().cpu().numpy()


def build(wl, step_tokens):
    """GPU cache after ctx_tokens + step_tokens tokens per sequence (the last
    step_tokens appended to every sequence by one batched call)."""
    caps = [(t + step_tokens) // wl.m + 8 for t in wl.ctx_tokens]
    cache = csa.Cache(caps, wl.d_idx, wl.m, DEV)
    for b, T in enumerate(wl.ctx_tokens):
        done = 0
        while done < T:
            n = min(1 << 17, T - done)
            C, Z = ci.latent_rows(wl, b, done, n, DEV)
            key = ci.key_rows(wl, b, done // wl.m, n // wl.m, DEV)
            csa.quantize_append(cache, C[None].contiguous(),
                                None if Z is None else Z[None].contiguous(),
                                key[None].contiguous(), seq=b)
            done += n
    if step_tokens:
        assert len(set(wl.ctx_tokens)) == 1
        T = wl.ctx_tokens[0]
        Cs, Zs, ks = [], [], []
        for b in range(wl.batch):
            C, Z = ci.latent_rows(wl, b, T, step_tokens, DEV)
            Cs.append(C)
            Zs.append(Z)
            ks.append(ci.key_rows(wl, b, T // wl.m, step_tokens // wl.m, DEV))
        csa.quantize_append(cache, torch.stack(Cs), None if wl.m == 1 else torch.stack(Zs),
                            torch.stack(ks))
    torch.cuda.synchronize()
    return cache


def oracle_keys(wl, b, n):
    return O.fp8_encode_rows(ci.key_rows(wl, b, 0, n, DEV).cpu().numpy())


def oracle_rows(wl, b, entries):
    C, Z = ci.latent_rows_at(wl, b, entries, DEV)
    C = C.reshape(1, -1, 512).cpu().numpy()
    Zn = None if Z is None else Z.reshape(1, -1, 512).cpu().numpy()
    key = np.zeros((1, len(entries), wl.d_idx), np.float32)
    codes, scales, _k, _s, _x, _ = O.append(C, Zn, key, wl.m)
    return codes, scales


def check_attention(wl, b, t, sel, qa, win, wcap, out_gpu):
    codes, scales = oracle_rows(wl, b, sel)
    rows = O.gather_rows(codes, scales, 0, np.arange(len(sel), dtype=np.int32),
                         bits16(win[b]), wcap, t, 0, wl.n_win)
    ref, _ = O.attention(bits16(qa), rows, wl.sm_scale)
    err = rel_rows(out_gpu, ref).max()
    assert err <= TOL, err


def test_decode_full_b32_ctx65536():
    """Decoder Full-mode decode: 32 sequences x 65,536 tokens, top-2048, 64 heads."""
    wl = ci.config(2, exact=True)
    T = wl.ctx_tokens[0]
    cache = build(wl, 1)
    B = wl.batch
    qs = csa.Queries(list(range(B)), [T] * B, 1, DEV)
    qi, w, qa = ci.query_inputs(wl, B, DEV)
    wcap = 256
    win = ci.window_rows(wl, B, wcap, DEV)
    idx = torch.zeros(B, wl.k, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(B, dtype=torch.int32, device=DEV)
    out = torch.zeros(B, wl.heads, 512, device=DEV)
    counters = csa.new_counters()
    csa.Layer(csa.FULL, cache, qs, k=wl.k, q=qa, win=win, n_win=wl.n_win, out=out, idx=idx,
              cnt=cnt, q_idx=qi, w=w, max_n=T + 1, counters=counters)()
    torch.cuda.synchronize()
    assert _np(counters).tolist() == [0, 0, 0, 0]
    n = T + 1
    for b in (0, 19, 31):
        k8, ks = oracle_keys(wl, b, n)
        sc = O.scores_full(k8, ks, _np(qi[b]), _np(w[b]), 0, n)
        ref = O.topk(sc, wl.k)
        assert int(cnt[b]) == wl.k and np.array_equal(_np(idx[b]), ref), b
        check_attention(wl, b, T, ref, qa[b], win, wcap, _np(out[b]))


def _near_kth(sc, got, ref, k):
    """Positions in which the GPU and oracle top-k sets differ, and whether each
    one's oracle score lies within 2e-3 * max|score| of the k-th largest oracle
    score (the only place where fp32 and float64 sums may disagree)."""
    diff = np.setxor1d(got, ref)
    kth = np.sort(sc)[::-1][min(k, len(sc)) - 1]
    tol = TOL * np.abs(sc).max()
    return diff, bool(np.all(np.abs(sc[diff] - kth) <= tol))


def test_decode_full_b32_ctx65536_random_float():
    """The same Full-mode decode with random-float indexer inputs (not exact in
    fp32): the GPU's fp32 scores may order near-equal candidates differently
    from the float64 oracle, so the two top-2048 sets may differ only among
    candidates whose oracle score is within 2e-3 * max|score| of the k-th
    score; the attention is then checked over the GPU's own selection."""
    wl = ci.config(2)
    T = wl.ctx_tokens[0]
    cache = build(wl, 1)
    B = wl.batch
    qs = csa.Queries(list(range(B)), [T] * B, 1, DEV)
    qi, w, qa = ci.query_inputs(wl, B, DEV)
    wcap = 256
    win = ci.window_rows(wl, B, wcap, DEV)
    idx = torch.zeros(B, wl.k, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(B, dtype=torch.int32, device=DEV)
    out = torch.zeros(B, wl.heads, 512, device=DEV)
    counters = csa.new_counters()
    csa.Layer(csa.FULL, cache, qs, k=wl.k, q=qa, win=win, n_win=wl.n_win, out=out, idx=idx,
              cnt=cnt, q_idx=qi, w=w, max_n=T + 1, counters=counters)()
    torch.cuda.synchronize()
    assert _np(counters).tolist() == [0, 0, 0, 0]
    n = T + 1
    n_diff = 0
    for b in (0, 7, 19, 31):
        k8, ks = oracle_keys(wl, b, n)
        sc = O.scores_full(k8, ks, _np(qi[b]), _np(w[b]), 0, n)
        ref = O.topk(sc, wl.k)
        got = _np(idx[b])
        assert int(cnt[b]) == wl.k and np.all(np.diff(got) > 0), b
        diff, near = _near_kth(sc, got, ref, wl.k)
        assert near, (b, diff)
        n_diff += len(diff) // 2
        check_attention(wl, b, T, got, qa[b], win, wcap, _np(out[b]))
    print(f"random-float top-{wl.k}: {n_diff} swapped candidates over 4 queries (all near the k-th score)")


def test_decode_reindex_b8_ctx1m():
    """A Full layer at 1M context builds the 2,048-block pool (16,384
    positions); a Reindex layer rescores only the pool; a Reuse layer follows."""
    wl = ci.config(3, exact=True)
    T = wl.ctx_tokens[0]
    cache = build(wl, 1)
    B = wl.batch
    n = T + 1
    qs = csa.Queries(list(range(B)), [T] * B, 1, DEV)
    wcap = 256
    pool_blk = torch.zeros(B, 2048, dtype=torch.int32, device=DEV)
    pool_n = torch.zeros(B, dtype=torch.int32, device=DEV)
    L = []
    for layer in range(3):
        qi, w, qa = ci.query_inputs(wl, B, DEV, layer=layer)
        L.append(dict(qi=qi, w=w, qa=qa, win=ci.window_rows(wl, B, wcap, DEV, layer=layer),
                      out=torch.zeros(B, wl.heads, 512, device=DEV)))
    idx_f = torch.zeros(B, wl.k, dtype=torch.int32, device=DEV)
    cnt_f = torch.zeros(B, dtype=torch.int32, device=DEV)
    idx_r = torch.zeros(B, wl.k, dtype=torch.int32, device=DEV)
    cnt_r = torch.zeros(B, dtype=torch.int32, device=DEV)
    counters = csa.new_counters()
    csa.Layer(csa.FULL, cache, qs, k=wl.k, q=L[0]["qa"], win=L[0]["win"], n_win=wl.n_win,
              out=L[0]["out"], idx=idx_f, cnt=cnt_f, q_idx=L[0]["qi"], w=L[0]["w"], max_n=n,
              build_pool=True, pool_blk=pool_blk, pool_n=pool_n, counters=counters)()
    csa.Layer(csa.REINDEX, cache, qs, k=wl.k, q=L[1]["qa"], win=L[1]["win"], n_win=wl.n_win,
              out=L[1]["out"], idx=idx_r, cnt=cnt_r, q_idx=L[1]["qi"], w=L[1]["w"], max_n=n,
              pool_blk=pool_blk, pool_n=pool_n, counters=counters)()
    csa.Layer(csa.REUSE, cache, qs, k=wl.k, q=L[2]["qa"], win=L[2]["win"], n_win=wl.n_win,
              out=L[2]["out"], idx=idx_r, cnt=cnt_r, max_n=n, counters=counters)()
    torch.cuda.synchronize()
    assert _np(counters).tolist() == [0, 0, 0, 0]
    assert _np(pool_n).tolist() == [16384] * B            # 2,048 x 8 ([Notes] section 3)
    b = 5
    k8, ks = oracle_keys(wl, b, n)
    sc = O.scores_full(k8, ks, _np(L[0]["qi"][b]), _np(L[0]["w"][b]), 0, n)
    ref_f = O.topk(sc, wl.k)
    assert np.array_equal(_np(idx_f[b]), ref_f)
    blk, pn = O.pool(sc, 2048)
    assert pn == 16384 and np.array_equal(_np(pool_blk[b]), blk)
    pos = (8 * blk[:, None] + np.arange(8)[None]).reshape(-1)
    sc_r = O.scores_at(k8, ks, _np(L[1]["qi"][b]), _np(L[1]["w"][b]), pos.astype(np.int64))
    ref_r = O.topk(sc_r, wl.k, pos.astype(np.int32))
    assert np.array_equal(_np(idx_r[b]), ref_r)
    check_attention(wl, b, T, ref_f, L[0]["qa"][b], L[0]["win"], wcap, _np(L[0]["out"][b]))
    check_attention(wl, b, T, ref_r, L[1]["qa"][b], L[1]["win"], wcap, _np(L[1]["out"][b]))
    check_attention(wl, b, T, ref_r, L[2]["qa"][b], L[2]["win"], wcap, _np(L[2]["out"][b]))


def test_prefill_m2_prefix262144_q4096():
    """Encoder prefill chunk: 4,096 causal queries appended to a 262,144-token
    prefix at m = 2 (131,072 + 2,048 entries); one Full + five Reuse layers.
    Latents on a 2^-10 grid with Z equal per block make the compression exact,
    so both sides hold the same FP4 cache."""
    wl = ci.config(4, exact=True, grid=True, equal_z=True, rms_norm=False)
    P = wl.ctx_tokens[0]
    nq = wl.q_per_seq
    cache = build(wl, nq)
    q_pos = [P + i for i in range(nq)]
    qs = csa.Queries([0] * nq, q_pos, wl.group, DEV)
    wcap = 8192
    n_max = (P + nq) // 2
    idx = torch.zeros(nq, wl.k, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(nq, dtype=torch.int32, device=DEV)
    counters = csa.new_counters()
    layers = []
    for layer in range(6):
        qi, w, qa = ci.query_inputs(wl, nq, DEV, layer=layer)
        win = ci.window_rows(wl, 1, wcap, DEV, layer=layer)
        out = torch.zeros(nq, wl.heads, 512, device=DEV)
        mode = csa.FULL if layer == 0 else csa.REUSE
        csa.Layer(mode, cache, qs, k=wl.k, q=qa, win=win, n_win=wl.n_win, out=out, idx=idx,
                  cnt=cnt, q_idx=qi if layer == 0 else None, w=w if layer == 0 else None,
                  max_n=n_max, counters=counters)()
        layers.append(dict(qi=qi, w=w, qa=qa, win=win, out=out))
    torch.cuda.synchronize()
    assert _np(counters).tolist() == [0, 0, 0, 0]
    k8, ks = oracle_keys(wl, 0, n_max)
    for i in (0, 1001, 4095):
        n = (q_pos[i] + 1) // 2
        sc = O.scores_full(k8, ks, _np(layers[0]["qi"][i]), _np(layers[0]["w"][i]), 0, n)
        ref = O.topk(sc, wl.k)
        assert int(cnt[i]) == wl.k and np.array_equal(_np(idx[i]), ref), i
        for layer in (0, 3, 5):
            Ly = layers[layer]
            check_attention(wl, 0, q_pos[i], ref, Ly["qa"][i], Ly["win"], wcap, _np(Ly["out"][i]))


def test_decoder_schedule_20_layers_mixed_lengths():
    """The 20-layer decoder (1 Full + 4 Reindex + 15 Reuse) over 64 sequences
    with log-uniform contexts in [4,096, 1,048,576], one new token each."""
    base = ci.config(5, exact=True)
    lens = base.ctx_tokens
    wl = ci.Workload(base.name, base.batch, lens, 0, 1, exact=True, rms_norm=True, seed=base.seed)
    caps = [t + 1 + 8 for t in lens]
    cache = csa.Cache(caps, wl.d_idx, wl.m, DEV)
    for b, T in enumerate(lens):
        done = 0
        while done < T + 1:              # context plus the step's new token
            n = min(1 << 17, T + 1 - done)
            C, _ = ci.latent_rows(wl, b, done, n, DEV)
            key = ci.key_rows(wl, b, done, n, DEV)
            csa.quantize_append(cache, C[None].contiguous(), None, key[None].contiguous(), seq=b)
            done += n
    torch.cuda.synchronize()
    B = wl.batch
    q_pos = list(lens)
    qs = csa.Queries(list(range(B)), q_pos, 1, DEV)
    wcap = 256
    per_layer = []
    for layer in range(20):
        qi, w, qa = ci.query_inputs(wl, B, DEV, layer=layer)
        per_layer.append(dict(q_idx=qi, w=w, q=qa, win=ci.window_rows(wl, B, wcap, DEV, layer=layer),
                              out=torch.zeros(B, wl.heads, 512, device=DEV)))
    counters = csa.new_counters()
    step = S.DecoderStep(csa, cache, qs, per_layer, k=wl.k, n_win=wl.n_win,
                         max_n=max(q_pos) + 1, counters=counters)
    step()
    torch.cuda.synchronize()
    assert _np(counters).tolist() == [0, 0, 0, 0]
    plan = S.decoder_schedule()
    for b in (int(np.argmin(lens)), int(np.argsort(lens)[B // 2])):
        n = q_pos[b] + 1
        k8, ks = oracle_keys(wl, b, n)
        L0 = per_layer[0]
        sc = O.scores_full(k8, ks, _np(L0["q_idx"][b]), _np(L0["w"][b]), 0, n)
        sel = {1: O.topk(sc, wl.k)}
        blk, pn = O.pool(sc, 2048)
        assert int(step.pool_n[b]) == pn
        assert np.array_equal(_np(step.pool_blk[b])[:len(blk)], blk)
        pos = np.array([8 * blk[p // 8] + p % 8 for p in range(pn)], np.int64)
        for p in plan:
            Ly = per_layer[p.layer - 1]
            if p.mode == S.REINDEX:
                scr = O.scores_at(k8, ks, _np(Ly["q_idx"][b]), _np(Ly["w"][b]), pos)
                sel[p.layer] = O.topk(scr, wl.k, pos.astype(np.int32))
            src = p.layer if p.mode != S.REUSE else p.source
            if p.mode != S.REUSE:
                got = _np(step.idx[src][b])[:int(step.cnt[src][b])]
                assert np.array_equal(got, sel[src]), (b, p.layer)
            if p.layer in (1, 4, 5, 20):
                check_attention(wl, b, q_pos[b], sel[src], Ly["q"][b], Ly["win"], wcap,
                                _np(Ly["out"][b]))


def test_encoder_chunk_18_layers_three_caches():
    """The encoder's 18 CSA2 layers (three blocks of 1 Full + 5 Reuse at m = 2)
    over one chunk of 64 causal queries after a 16,000-token prefix, each block
    with its own cache; exact-integer indexer inputs and exactly compressible
    latents, as in the prefill test."""
    P, nq = 16000, 64
    wls = [ci.Workload(f"enc{b}", 1, [P], nq, 2, exact=True, grid=True, equal_z=True,
                       seed=1100 + b, group=32, q_per_seq=nq) for b in range(3)]
    caches = [build(wl, nq) for wl in wls]
    q_pos = [P + i for i in range(nq)]
    qs = csa.Queries([0] * nq, q_pos, 32, DEV)
    wcap = 512
    n_max = (P + nq) // 2
    plan = S.encoder_csa2_layers()
    per_layer = []
    for i, p in enumerate(plan):
        wl = wls[p.cache]
        qi, w, qa = ci.query_inputs(wl, nq, DEV, layer=i)
        per_layer.append(dict(q_idx=qi, w=w, q=qa, win=ci.window_rows(wl, 1, wcap, DEV, layer=i),
                              out=torch.zeros(nq, wl.heads, 512, device=DEV)))
    counters = csa.new_counters()
    chunk = S.EncoderChunk(csa, caches, qs, per_layer, k=wls[0].k, n_win=wls[0].n_win,
                           max_n=n_max, counters=counters)
    chunk()
    torch.cuda.synchronize()
    assert _np(counters).tolist() == [0, 0, 0, 0]
    for b in range(3):
        wl = wls[b]
        k8, ks = oracle_keys(wl, 0, n_max)
        lay = [i for i, p in enumerate(plan) if p.cache == b]
        full = per_layer[lay[0]]
        for i in (0, 37, 63):
            n = (q_pos[i] + 1) // 2
            sc = O.scores_full(k8, ks, _np(full["q_idx"][i]), _np(full["w"][i]), 0, n)
            ref = O.topk(sc, wl.k)
            assert int(chunk.cnt[b][i]) == wl.k and np.array_equal(_np(chunk.idx[b][i]), ref), (b, i)
            for j in (lay[0], lay[2], lay[5]):           # the Full layer and two Reuse layers
                Ly = per_layer[j]
                check_attention(wl, 0, q_pos[i], ref, Ly["q"][i], Ly["win"], wcap, _np(Ly["out"][i]))
