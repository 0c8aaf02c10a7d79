"""Parity of each CUDA entry point with the float64 oracle, at sizes the oracle
finishes in seconds that still span several tiles and a ragged tail.

Bars: FP4 codes/scales and FP8 keys bit-exact; top-k indices and pools
bit-exact on identical score arrays and end to end in exact-integer mode;
scores and attention outputs within 2e-3 of the row's max |oracle| value."""
import numpy as np
import pytest
import torch

import csa2_inputs as ci
import oracle as O
import sparse_attention_decode_step_gb300 as csa
from helpers import (TOL, bits16, build_gpu_cache, need_gpu, oracle_rows, oracle_seq_cache,
                     rel_rows)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _gpu():
    need_gpu()


def _np(t):
    return t.detach().cpu().numpy()


# ================================================================ append
@pytest.mark.parametrize("d_idx", [128, 64])
def test_append_m1_bit_exact(d_idx):
    wl = ci.Workload("t", 3, [1000, 333, 7], 0, 1, d_idx=d_idx, seed=11)
    cnt = csa.new_counters()
    cache = build_gpu_cache(wl, DEV, counters=cnt)
    torch.cuda.synchronize()
    assert _np(cache.seq_len).tolist() == [1000, 333, 7]
    assert _np(cnt).tolist() == [0, 0, 0, 0]
    for b, n in enumerate([1000, 333, 7]):
        codes, scales, kidx, ksc, _ = oracle_rows(wl, b, 0, n)
        r0 = cache.base_host[b]
        assert np.array_equal(_np(cache.codes[r0:r0 + n]), codes)
        assert np.array_equal(_np(cache.scales[r0:r0 + n]), scales)
        assert np.array_equal(_np(cache.kidx[r0:r0 + n]), kidx)
        assert np.array_equal(_np(cache.kscale[r0:r0 + n]), ksc)


def test_append_batched_call_and_growth():
    # one call appends to every sequence; a second call continues after it
    wl = ci.Workload("t", 2, [0, 0], 0, 1, seed=12)
    cache = csa.Cache([64, 64], 128, 1, DEV)
    C = torch.stack([ci.latent_rows(wl, b, 0, 24, DEV)[0] for b in range(2)])
    key = torch.stack([ci.key_rows(wl, b, 0, 24, DEV) for b in range(2)])
    csa.quantize_append(cache, C[:, :10].contiguous(), None, key[:, :10].contiguous())
    csa.quantize_append(cache, C[:, 10:].contiguous(), None, key[:, 10:].contiguous())
    torch.cuda.synchronize()
    assert _np(cache.seq_len).tolist() == [24, 24]
    for b in range(2):
        codes, scales, kidx, ksc, _ = oracle_rows(wl, b, 0, 24)
        r0 = cache.base_host[b]
        assert np.array_equal(_np(cache.codes[r0:r0 + 24]), codes)
        assert np.array_equal(_np(cache.kidx[r0:r0 + 24]), kidx)


def test_append_m2_exact_inputs_bit_exact():
    # equal Z -> weights exactly 1/2; latents on a 2^-10 grid -> the block mean is exact in fp32
    B, n_tok = 2, 64
    g = torch.Generator().manual_seed(3)
    C = (torch.randint(-4096, 4097, (B, n_tok, 512), generator=g).float() / 1024.0)
    Z = torch.randn(B, n_tok // 2, 1, 512, generator=g).expand(B, n_tok // 2, 2, 512).reshape(B, n_tok, 512)
    key = torch.randn(B, n_tok // 2, 128, generator=g)
    cache = csa.Cache([64, 64], 128, 2, DEV)
    csa.quantize_append(cache, C.to(DEV), Z.contiguous().to(DEV), key.to(DEV))
    torch.cuda.synchronize()
    codes, scales, kidx, ksc, x, _ = O.append(C.numpy(), Z.contiguous().numpy(), key.numpy(), 2)
    for b in range(B):
        r0 = cache.base_host[b]
        sl = slice(b * 32, b * 32 + 32)
        assert np.array_equal(_np(cache.codes[r0:r0 + 32]), codes[sl])
        assert np.array_equal(_np(cache.scales[r0:r0 + 32]), scales[sl])
        assert np.array_equal(_np(cache.kidx[r0:r0 + 32]), kidx[sl])


def test_append_m2_random_differs_only_at_rounding_boundaries():
    wl = ci.Workload("t", 1, [4096], 0, 2, d_idx=64, seed=13)
    cache = build_gpu_cache(wl, DEV)
    torch.cuda.synchronize()
    n = 2048
    codes, scales, kidx, ksc, x = oracle_rows(wl, 0, 0, n)
    gc, gs = _np(cache.codes[:n]), _np(cache.scales[:n])
    assert np.array_equal(_np(cache.kidx[:n]), kidx)
    ok_scale = gs == scales
    for r, g in np.argwhere(~ok_scale):
        # a different scale only where amax / 6 sits on an E4M3 value (fp32 vs fp64 edge)
        amax = np.abs(x[r, 16 * g:16 * g + 16]).max()
        edge = 6.0 * min(O.e4m3_value(int(gs[r, g])), O.e4m3_value(int(scales[r, g])))
        assert abs(amax - edge) <= 1e-5 * amax, (r, g)
    assert (~ok_scale).sum() <= 2
    dg = O.fp4_decode_rows(gc, gs)
    do = O.fp4_decode_rows(codes, scales)
    same_scale = np.repeat(ok_scale, 16, axis=1)
    diff = np.argwhere((dg != do) & same_scale)
    assert len(diff) <= n * 512 * 1e-3
    for r, c in diff:
        # the fp64 value sits on the rounding midpoint the fp32 value fell across
        mid = 0.5 * (dg[r, c] + do[r, c])
        assert abs(x[r, c] - mid) <= 1e-5 * abs(mid), (r, c, x[r, c], dg[r, c], do[r, c])


def _bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


@pytest.mark.parametrize("d_idx,m", [(128, 1), (64, 1), (128, 2)])
def test_append_project_exact_inputs_bit_exact(d_idx, m):
    # integer latents in [-6, 6] with a 6 in every group (all scales 1.0; at m = 2
    # equal Z makes each entry the exact mean of its two tokens) and W_IK entries
    # k / 64: the projected keys are exact in fp32, so every byte matches.
    # 4 sequences x 8 tokens (decode-sized) and one sequence of 3,000 tokens
    # (many entries per warp)
    g = torch.Generator().manual_seed(44)
    w = _bf16(torch.randint(-64, 65, (512, d_idx), generator=g) / 64.0)
    wbits = w.view(torch.int16).numpy().view(np.uint16)
    for B, n_tok in ((4, 8), (1, 3000)):
        C = torch.randint(-6, 7, (B, n_tok, 512), generator=g).float()
        C[..., ::16] = 6.0
        Z = None
        if m == 2:
            Z = torch.randn(B, n_tok // 2, 1, 512, generator=g).expand(B, n_tok // 2, 2, 512)
            Z = Z.reshape(B, n_tok, 512).contiguous()
        ne = n_tok // m
        cache = csa.Cache([ne + 8] * B, d_idx, m, DEV)
        cnt = csa.new_counters()
        csa.quantize_append_project(cache, C.to(DEV), None if Z is None else Z.to(DEV), w.to(DEV),
                                    counters=cnt)
        torch.cuda.synchronize()
        assert _np(cache.seq_len).tolist() == [ne] * B and _np(cnt).tolist() == [0, 0, 0, 0]
        codes, scales, kidx, ksc, _k, _ = O.append_project(C.numpy(),
                                                           None if Z is None else Z.numpy(), wbits, m)
        for b in range(B):
            r0, sl = cache.base_host[b], slice(b * ne, (b + 1) * ne)
            assert np.array_equal(_np(cache.codes[r0:r0 + ne]), codes[sl])
            assert np.array_equal(_np(cache.scales[r0:r0 + ne]), scales[sl])
            assert np.array_equal(_np(cache.kidx[r0:r0 + ne]), kidx[sl])
            assert np.array_equal(_np(cache.kscale[r0:r0 + ne]), ksc[sl])


def test_append_project_random_differs_only_at_rounding_boundaries():
    # random latents and W_IK (m = 1: the FP4 entries are bit-exact for any
    # input); each key byte matches the oracle unless the fp64 key sits on the
    # E4M3 rounding midpoint that the fp32 sum fell across
    g = torch.Generator().manual_seed(45)
    B, n_tok, d_idx = 2, 512, 128
    C = torch.randn(B, n_tok, 512, generator=g)
    w = _bf16(torch.randn(512, d_idx, generator=g) / 16.0)
    cache = csa.Cache([n_tok + 8] * B, d_idx, 1, DEV)
    csa.quantize_append_project(cache, C.to(DEV), None, w.to(DEV))
    torch.cuda.synchronize()
    wbits = w.view(torch.int16).numpy().view(np.uint16)
    codes, scales, kidx, ksc, k, _ = O.append_project(C.numpy(), None, wbits, 1)
    ne = n_tok
    gc = np.concatenate([_np(cache.codes[cache.base_host[b]:cache.base_host[b] + ne]) for b in range(B)])
    gs = np.concatenate([_np(cache.scales[cache.base_host[b]:cache.base_host[b] + ne]) for b in range(B)])
    gk = np.concatenate([_np(cache.kidx[cache.base_host[b]:cache.base_host[b] + ne]) for b in range(B)])
    gks = np.concatenate([_np(cache.kscale[cache.base_host[b]:cache.base_host[b] + ne]) for b in range(B)])
    assert np.array_equal(gc, codes) and np.array_equal(gs, scales)
    rows = np.arange(B * ne)
    assert np.array_equal(gks[rows], ksc[rows])   # no amax on a power-of-two edge here
    tab = O.e4m3_values(np.arange(256))
    y = k[rows] / ksc[rows, None]
    diff = np.argwhere(gk[rows] != kidx[rows])
    assert len(diff) <= 1e-3 * y.size
    for r, c in diff:
        a, b_ = tab[gk[rows][r, c]], tab[kidx[rows][r, c]]
        mid = 0.5 * (a + b_)
        assert abs(y[r, c] - mid) <= 1e-5 * max(1.0, abs(mid)), (r, c, y[r, c], a, b_)


def test_append_saturation_and_capacity_counters():
    cache = csa.Cache([16], 128, 1, DEV)
    C = torch.zeros(1, 8, 512)
    C[0, 0, :16] = 3000.0          # one saturated group
    C[0, 3, 100] = -5000.0         # another
    key = torch.ones(1, 8, 128)
    cnt = csa.new_counters()
    csa.quantize_append(cache, C.to(DEV), None, key.to(DEV), counters=cnt)
    csa.quantize_append(cache, C.to(DEV), None, key.to(DEV), counters=cnt)
    csa.quantize_append(cache, C.to(DEV), None, key.to(DEV), counters=cnt)   # 24 > 16: refused
    torch.cuda.synchronize()
    assert _np(cnt).tolist() == [4, 1, 0, 0]
    assert int(cache.seq_len[0]) == 16
    codes, scales, _k, _s, _x, nsat = O.append(C.numpy(), None, key.numpy(), 1)
    assert nsat == 2
    assert np.array_equal(_np(cache.codes[:8]), codes) and np.array_equal(_np(cache.scales[8:16]), scales)


# ================================================================ indexer
def _index_case(wl, lengths, positions, exact):
    cache = build_gpu_cache(wl, DEV)
    q_seq = [b for b, _ in positions]
    q_pos = [t for _, t in positions]
    qs = csa.Queries(q_seq, q_pos, 1, DEV)
    qi, w, _qa = ci.query_inputs(wl, len(q_seq), "cpu")
    max_n = max(lengths)
    ld = (max_n + 3) // 4 * 4
    scores = torch.full((len(q_seq), ld), float("nan"), device=DEV)
    bm = torch.full((len(q_seq), ((max_n + 7) // 8 + 3) // 4 * 4), float("nan"), device=DEV)
    nv = torch.zeros(len(q_seq), dtype=torch.int32, device=DEV)
    cnt = csa.new_counters()
    csa.index_full(cache, qs, qi.to(DEV), w.to(DEV), max_n, scores, blockmax=bm, n_valid=nv,
                   counters=cnt)
    torch.cuda.synchronize()
    assert _np(cnt).tolist() == [0, 0, 0, 0]
    gs, gb = _np(scores), _np(bm)
    for i, (b, t) in enumerate(positions):
        n = (t + 1) // wl.m
        assert int(nv[i]) == n
        oc = oracle_seq_cache(wl, b, n)
        ref = O.scores_full(oc["kidx"], oc["kscale"], qi[i].numpy(), w[i].numpy(), 0, n)
        refbm = O.blockmax(ref)
        if exact:
            assert np.array_equal(gs[i, :n].astype(np.float64), ref), i
            assert np.array_equal(gb[i, :(n + 7) // 8].astype(np.float64), refbm), i
        else:
            assert rel_rows(gs[i, :n][None], ref[None])[0] <= TOL
            assert rel_rows(gb[i, :(n + 7) // 8][None], refbm[None])[0] <= TOL


@pytest.mark.parametrize("exact", [True, False])
def test_index_full_ragged_batch(exact):
    lengths = [5000, 130, 1029]
    wl = ci.Workload("t", 3, lengths, 0, 1, exact=exact, seed=21)
    positions = [(0, 4999), (1, 129), (2, 1028), (0, 2047), (2, 7), (0, 0)]
    _index_case(wl, lengths, positions, exact)


def test_index_full_tiny_shape_m2():
    # d_idx 64, 4 indexer heads, m = 2 (tiny workload shape)
    wl = ci.Workload("t", 1, [4096], 0, 2, h_idx=4, d_idx=64, exact=True, seed=22)
    _index_case(wl, [2048], [(0, 4095), (0, 4094), (0, 1001)], True)


@pytest.mark.parametrize("exact", [True, False])
def test_index_full_grouped_prefill(exact):
    # 64 causal queries of one sequence scored together (groups of 32, N = 256)
    wl = ci.Workload("t", 1, [6000], 0, 2, exact=exact, seed=23)
    cache = build_gpu_cache(wl, DEV)
    nq = 64
    q_pos = [5936 + i for i in range(nq)]
    qs = csa.Queries([0] * nq, q_pos, 32, DEV)
    qi, w, _ = ci.query_inputs(wl, nq, "cpu")
    max_n = 3000
    scores = torch.full((nq, max_n), float("nan"), device=DEV)
    bm = torch.full((nq, (max_n // 8 + 3) // 4 * 4), float("nan"), device=DEV)
    csa.index_full(cache, qs, qi.to(DEV), w.to(DEV), max_n, scores, blockmax=bm)
    torch.cuda.synchronize()
    oc = oracle_seq_cache(wl, 0, 3000)
    gs, gb = _np(scores), _np(bm)
    for i in range(nq):
        n = (q_pos[i] + 1) // 2
        ref = O.scores_full(oc["kidx"], oc["kscale"], qi[i].numpy(), w[i].numpy(), 0, n)
        if exact:
            assert np.array_equal(gs[i, :n].astype(np.float64), ref), i
            assert np.array_equal(gb[i, :(n + 7) // 8].astype(np.float64), O.blockmax(ref)), i
        else:
            assert rel_rows(gs[i, :n][None], ref[None])[0] <= TOL


@pytest.mark.parametrize("group,h_idx,d_idx", [(10, 8, 128), (6, 16, 64), (4, 4, 128)])
def test_index_full_groups_uneven_column_halves(group, h_idx, d_idx):
    # N = group * h_idx = 80 and 96: the two-CTA launch whose eight epilogue warps
    # split the columns unevenly (64 + 16, 64 + 32; the second half's MMA is
    # N = 16 or 32 and its B operand starts mid-tile); N = 16: a small group
    # in the one-CTA launch.  Exact integer inputs: scores bit-exact.
    wl = ci.Workload("t", 1, [6000], 0, 2, h_idx=h_idx, d_idx=d_idx, exact=True, seed=25)
    cache = build_gpu_cache(wl, DEV)
    nq = 2 * group
    q_pos = [5960 - 3 * i for i in range(nq)]
    qs = csa.Queries([0] * nq, q_pos, group, DEV)
    qi, w, _ = ci.query_inputs(wl, nq, "cpu")
    max_n = 3000
    scores = torch.full((nq, max_n), float("nan"), device=DEV)
    bm = torch.full((nq, (max_n // 8 + 3) // 4 * 4), float("nan"), device=DEV)
    csa.index_full(cache, qs, qi.to(DEV), w.to(DEV), max_n, scores, blockmax=bm)
    torch.cuda.synchronize()
    oc = oracle_seq_cache(wl, 0, 3000)
    gs, gb = _np(scores), _np(bm)
    for i in range(nq):
        n = (q_pos[i] + 1) // 2
        ref = O.scores_full(oc["kidx"], oc["kscale"], qi[i].numpy(), w[i].numpy(), 0, n)
        assert np.array_equal(gs[i, :n].astype(np.float64), ref), i
        assert np.array_equal(gb[i, :(n + 7) // 8].astype(np.float64), O.blockmax(ref)), i


@pytest.mark.parametrize("exact", [True, False])
def test_index_reindex_pool(exact):
    n = 20000
    wl = ci.Workload("t", 2, [n, 9000], 0, 1, exact=exact, seed=24)
    cache = build_gpu_cache(wl, DEV)
    rng = np.random.default_rng(5)
    pool_blocks = 2048
    blk0 = np.sort(rng.choice(n // 8, 2048, replace=False)).astype(np.int32)
    blk1 = np.sort(rng.choice(9000 // 8, 700, replace=False)).astype(np.int32)
    pool = np.zeros((2, pool_blocks), np.int32)
    pool[0] = blk0
    pool[1, :700] = blk1
    pool_n = np.array([8 * 2048, 8 * 700 - 3], np.int32)     # ragged tail on query 1
    qs = csa.Queries([0, 1], [n - 1, 8999], 1, DEV)
    qi, w, _ = ci.query_inputs(wl, 2, "cpu")
    scores = torch.full((2, 8 * pool_blocks), float("nan"), device=DEV)
    nv = torch.zeros(2, dtype=torch.int32, device=DEV)
    csa.index_reindex(cache, qs, qi.to(DEV), w.to(DEV), torch.from_numpy(pool).to(DEV),
                      torch.from_numpy(pool_n).to(DEV), scores, n_valid=nv)
    torch.cuda.synchronize()
    gs = _np(scores)
    for i, (nn, pn) in enumerate([(n, pool_n[0]), (9000, pool_n[1])]):
        assert int(nv[i]) == pn
        oc = oracle_seq_cache(wl, i, nn)
        rows = np.array([8 * pool[i, p // 8] + p % 8 for p in range(pn)], np.int64)
        ref = O.scores_at(oc["kidx"], oc["kscale"], qi[i].numpy(), w[i].numpy(), rows)
        if exact:
            assert np.array_equal(gs[i, :pn].astype(np.float64), ref)
        else:
            assert rel_rows(gs[i, :pn][None], ref[None])[0] <= TOL


def test_index_counts_query_past_cache():
    wl = ci.Workload("t", 1, [100], 0, 1, seed=25)
    cache = build_gpu_cache(wl, DEV)
    qs = csa.Queries([0, 0], [99, 150], 1, DEV)          # second query: position not cached
    qi, w, _ = ci.query_inputs(wl, 2, "cpu")
    scores = torch.zeros(2, 256, device=DEV)
    nv = torch.zeros(2, dtype=torch.int32, device=DEV)
    cnt = csa.new_counters()
    csa.index_full(cache, qs, qi.to(DEV), w.to(DEV), 256, scores, n_valid=nv, counters=cnt)
    torch.cuda.synchronize()
    assert int(cnt[csa.CNT_BAD_INPUT]) == 1 and _np(nv).tolist() == [100, 0]


# ================================================================ top-k and pool
def _topk_gpu(scores_np, nvalid, k, pool=None, ld=None):
    nq, n = scores_np.shape
    ld = ld or (n + 3) // 4 * 4
    s = torch.zeros(nq, ld, dtype=torch.float32)
    s[:, :n] = torch.from_numpy(scores_np)
    idx = torch.full((nq, k), -1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(nq, dtype=torch.int32, device=DEV)
    csa.topk(s.to(DEV), torch.tensor(nvalid, dtype=torch.int32, device=DEV), k, idx, cnt,
             max_n=n, pool_blk=None if pool is None else torch.from_numpy(pool).to(DEV))
    torch.cuda.synchronize()
    return _np(idx), _np(cnt)


@pytest.mark.parametrize("n,k", [(1, 1), (100, 7), (4096, 64), (4097, 4096), (70001, 2048),
                                 (73728, 4096), (73729, 2048), (20000, 5000), (300, 2048),
                                 (16384, 2048)])
def test_topk_bit_exact(n, k):
    rng = np.random.default_rng(n + k)
    s = rng.normal(size=(3, n)).astype(np.float32)
    s[1] = np.round(s[1] * 4) / 4                       # heavy ties
    s[2, ::7] = 0.0
    s[2, 3::7] = -0.0                                   # -0 equals +0
    nvalid = [n, max(1, n - 5), max(1, n // 3)]
    idx, cnt = _topk_gpu(s, nvalid, k)
    for i in range(3):
        ref = O.topk(s[i, :nvalid[i]], k)
        assert cnt[i] == len(ref)
        assert np.array_equal(idx[i, :cnt[i]], ref), i


@pytest.mark.parametrize("n", [50000, 65536])
def test_topk_all_equal_and_few_distinct(n):
    # every score equal (the k lowest positions win), and scores drawn from 3
    # values: tens of thousands of keys share every prefix of the radix rounds
    k = 2048
    s = np.full((2, n), 1.5, np.float32)
    rng = np.random.default_rng(n)
    s[1] = rng.choice(np.array([0.25, 1.0, 3.0], np.float32), size=n)
    idx, cnt = _topk_gpu(s, [n, n - 1], k)
    for i, nv in enumerate([n, n - 1]):
        ref = O.topk(s[i, :nv], k)
        assert cnt[i] == k and np.array_equal(idx[i, :k], ref), i


@pytest.mark.parametrize("n,k", [(70001, 2048), (262144, 2048), (9000, 4096)])
def test_topk_many_queries_bit_exact(n, k):
    # at least 96 queries in one call (a prefill chunk) take one CTA per query;
    # rows of every kind in one launch: random floats, heavy ties, all equal,
    # n <= k, three distinct values (the threshold bin exceeds the candidate
    # list), negative and positive zero, a ragged tail
    nq = 100
    rng = np.random.default_rng(n + 7 * k)
    s = rng.normal(size=(nq, n)).astype(np.float32)
    nvalid = []
    for i in range(nq):
        kind = i % 6
        if kind == 1:
            s[i] = np.round(s[i] * 4) / 4
        elif kind == 2:
            s[i] = 1.5
        elif kind == 4:
            s[i] = rng.choice(np.array([0.25, 1.0, 3.0], np.float32), size=n)
        elif kind == 5:
            s[i, ::5] = 0.0
            s[i, 2::5] = -0.0
        nvalid.append(int(rng.integers(1, k + 1)) if kind == 3 else n - int(rng.integers(0, 40)))
    idx, cnt = _topk_gpu(s, nvalid, k)
    for i in range(nq):
        ref = O.topk(s[i, :nvalid[i]], k)
        assert cnt[i] == len(ref), i
        assert np.array_equal(idx[i, :cnt[i]], ref), i


def test_topk_with_pool_map():
    rng = np.random.default_rng(1)
    pool = np.sort(rng.choice(100000, 2048, replace=False)).astype(np.int32)[None].repeat(2, 0)
    pn = [16384, 16381]
    s = np.round(rng.normal(size=(2, 16384)) * 8).astype(np.float32) / 8
    idx, cnt = _topk_gpu(s, pn, 2048, pool=pool)
    for i in range(2):
        pos = np.array([8 * pool[i, p // 8] + p % 8 for p in range(pn[i])], np.int32)
        ref = O.topk(s[i, :pn[i]], 2048, pos)
        assert np.array_equal(idx[i, :cnt[i]], ref)


def test_topk_many_queries_with_pool_map():
    # the one-CTA-per-query top-k (at least 96 queries) maps pool positions to
    # cache positions through each query's pool blocks
    nq, npos = 100, 16384
    rng = np.random.default_rng(5)
    pool = np.stack([np.sort(rng.choice(200000, 2048, replace=False)) for _ in range(nq)]).astype(np.int32)
    pn = [npos - int(rng.integers(0, 8)) for _ in range(nq)]
    s = np.round(rng.normal(size=(nq, npos)) * 8).astype(np.float32) / 8
    idx, cnt = _topk_gpu(s, pn, 2048, pool=pool)
    for i in range(nq):
        pos = np.array([8 * pool[i, p_ // 8] + p_ % 8 for p_ in range(pn[i])], np.int32)
        ref = O.topk(s[i, :pn[i]], 2048, pos)
        assert np.array_equal(idx[i, :cnt[i]], ref), i


def test_pool_select_many_queries_bit_exact():
    # pool selection over block maxima (candidates = blocks) for 100 queries in
    # one call, so that the one-CTA-per-query top-k picks the blocks
    nq = 100
    rng = np.random.default_rng(11)
    ns = [int(rng.integers(20000, 140000)) for _ in range(nq)]
    nbmax = (max(ns) + 7) // 8
    bm = torch.full((nq, (nbmax + 3) // 4 * 4), -np.inf, dtype=torch.float32)
    refs = []
    for i, n in enumerate(ns):
        sc = rng.normal(size=n)
        sc[rng.integers(0, n, size=40)] = 6.0                   # ties among the largest maxima
        rb = O.blockmax(sc)
        bm[i, :len(rb)] = torch.from_numpy(rb.astype(np.float32))
        refs.append(O.pool(np.repeat(rb.astype(np.float32), 8)[:n].astype(np.float64), 2048))
    blk = torch.full((nq, 2048), -1, dtype=torch.int32, device=DEV)
    pn = torch.zeros(nq, dtype=torch.int32, device=DEV)
    csa.pool_select(bm.to(DEV), torch.tensor(ns, dtype=torch.int32, device=DEV), max(ns), blk, pn)
    torch.cuda.synchronize()
    gb, gp = _np(blk), _np(pn)
    for i, n in enumerate(ns):
        ref_blk, ref_pn = refs[i]
        c = min(2048, (n + 7) // 8)
        assert np.array_equal(gb[i, :c], ref_blk) and int(gp[i]) == ref_pn, i


@pytest.mark.parametrize("n", [50, 16384, 16387, 200003])
def test_pool_select_bit_exact(n):
    rng = np.random.default_rng(n)
    sc = rng.normal(size=n)
    sc[-1] = 40.0                                        # newest (maybe partial) block wins
    refbm = O.blockmax(sc)
    nb = len(refbm)
    bm = torch.zeros(1, (nb + 3) // 4 * 4, dtype=torch.float32)
    bm[0, :nb] = torch.from_numpy(refbm.astype(np.float32))
    blk = torch.full((1, 2048), -1, dtype=torch.int32, device=DEV)
    pn = torch.zeros(1, dtype=torch.int32, device=DEV)
    csa.pool_select(bm.to(DEV), torch.tensor([n], dtype=torch.int32, device=DEV), n, blk, pn)
    torch.cuda.synchronize()
    # the oracle sees the same fp32 block maxima (each repeated over its block)
    ref_blk, ref_pn = O.pool(np.repeat(refbm.astype(np.float32), 8)[:n].astype(np.float64), 2048)
    c = min(2048, nb)
    assert np.array_equal(_np(blk)[0, :c], ref_blk) and int(pn[0]) == ref_pn


# ================================================================ attention
def _attn_case(H, n_ent, cnts, n_win, wcap, win_start=None, sm=1.0, seed=31, bad=False):
    nq = len(cnts)
    wl = ci.Workload("t", nq, [n_ent] * nq, 0, 1, heads=H, seed=seed)
    cache = build_gpu_cache(wl, DEV)
    rng = np.random.default_rng(seed)
    k_max = max(max(cnts), 1)
    idx = np.zeros((nq, k_max), np.int32)
    for i, c in enumerate(cnts):
        idx[i, :c] = np.sort(rng.choice(n_ent, c, replace=False))
    if bad:
        idx[0, 0] = n_ent + 5
    _qi, _w, qa = ci.query_inputs(wl, nq, "cpu")
    win = ci.window_rows(wl, nq, wcap, "cpu")
    qs = csa.Queries(list(range(nq)), [n_ent - 1] * nq, 1, DEV)
    out = torch.full((nq, H, 512), float("nan"), device=DEV)
    lse = torch.full((nq, H), float("nan"), device=DEV)
    cnt = csa.new_counters()
    ws_t = None if win_start is None else torch.tensor(win_start, dtype=torch.int32, device=DEV)
    csa.sparse_attn(cache, qs, torch.from_numpy(idx).to(DEV),
                    torch.tensor(cnts, dtype=torch.int32, device=DEV), qa.to(DEV),
                    win.to(DEV) if n_win else None, n_win, out, lse=lse, win_start=ws_t,
                    sm_scale=sm, counters=cnt)
    torch.cuda.synchronize()
    go, gl = _np(out), _np(lse)
    for i in range(nq):
        codes, scales, _k, _s, _x = oracle_rows(wl, i, 0, n_ent)
        sel = idx[i, :cnts[i]]
        if bad and i == 0:
            sel = sel[1:]
        s = 0 if win_start is None else win_start[i]
        rows = O.gather_rows(codes, scales, 0, sel, bits16(win[i]) if n_win else None, wcap,
                             n_ent - 1, s, n_win)
        ref, rlse = O.attention(bits16(qa[i]), rows, sm)
        assert rel_rows(go[i], ref).max() <= TOL, i
        assert np.abs(gl[i] - rlse).max() <= 1e-3 * max(1.0, np.abs(rlse).max())
    return _np(cnt)


@pytest.mark.parametrize("H", [64, 16])
def test_attention_matches_oracle(H):
    c = _attn_case(H, 3000, [2048, 5, 0, 1000], 128, 256)
    assert c.tolist() == [0, 0, 0, 0]


# (queries, rows per query) that make the planner divide a query over 2 .. 16
# CTAs on a 152-SM GPU: the cluster merge at every size it uses, including
# the sizes above the portable 8 and those whose owners take two chunk slots
@pytest.mark.parametrize("nq,rows,splits", [(64, 2176, 2), (40, 2176, 3), (30, 2176, 5),
                                            (25, 2176, 6), (21, 1792, 7), (19, 2048, 8),
                                            (15, 2560, 10),
                                            (13, 1408, 11), (12, 1536, 12), (9, 2048, 16)])
def test_attention_cluster_sizes(nq, rows, splits):
    if torch.cuda.get_device_properties(0).multi_processor_count == 152:
        assert _attn_splits(nq, rows) == splits
    n_win = 128
    cnts = [rows - n_win - (i % 3) * 40 for i in range(nq)]   # the first query has the most rows
    c = _attn_case(64, 3000, cnts, n_win, 256, seed=nq)
    assert c.tolist() == [0, 0, 0, 0]


def test_attention_window_truncation_and_scale():
    _attn_case(64, 600, [300, 17], 128, 128, win_start=[560, 0], sm=0.37, seed=32)


def test_attention_counts_and_skips_bad_index():
    c = _attn_case(32, 500, [40, 40], 16, 32, seed=33, bad=True)
    assert c[csa.CNT_BAD_INPUT] == 1


def test_attention_one_query_long_selection():
    # One query, 8000 selected rows plus 128 window rows: 64 row tiles (the
    # last one ragged) divided over the 8 CTAs of one cluster.
    _attn_case(64, 10000, [8000], 128, 256, seed=34)


def test_attention_more_queries_than_sms_single_split():
    # More queries than SMs: each query is one CTA (no cluster merge), with
    # empty, short and several-tile selections mixed.
    rng = np.random.default_rng(35)
    cnts = rng.integers(0, 257, size=156).tolist()
    cnts[:3] = [0, 256, 1]
    _attn_case(64, 256, cnts, 32, 64, seed=35)


# ---------------------------------------------------------------- peaky attention
# The kernel keeps, per head, a reference max that moves only when a tile's
# logit exceeds it by more than 8 (log2 units); the output accumulator is then
# rescaled in tensor memory.  A query's tile range may be split over up to 8
# CTAs whose partial results are merged with weights 2^(m_split - M).  The
# cases below make both paths run: heads whose logits spread over tens of log2
# units (q scaled by 16), heads whose winning row sits in a late tile of a
# late split or in an early split (the other splits' weights underflow), and
# heads whose winning row is a window row.
LOG2E = 1.4426950408889634


def _attn_splits(nq, n_rows_max, cap=16):
    """The number of CTAs per query the library uses (the rule of its planner,
    on a GPU that schedules clusters of 16): at most sms / nq, the tiles and
    the cap, 13 .. 15 skipped, then as few as give the same tiles per split."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = (n_rows_max + 127) // 128
    s = max(1, min(sms // nq, tiles, cap))
    if 12 < s < 16:
        s = 12
    tps = (tiles + s - 1) // s
    s = (tiles + tps - 1) // tps
    return 16 if 12 < s < 16 else s


def _split_tiles(n_rows, splits):
    """Row ranges of the 128-row tiles of each split (ceil division of the tiles)."""
    tiles = (n_rows + 127) // 128
    tps = (tiles + splits - 1) // splits
    out = []
    for s in range(splits):
        t0, t1 = min(tiles, s * tps), min(tiles, s * tps + tps)
        out.append([(128 * t, min(n_rows, 128 * t + 128)) for t in range(t0, t1)])
    return out


def _sel_rows(wl, b, sel, win_bits, wcap, t, n_win):
    """The oracle's row set of one query: its selected entries (encoded from the
    generator's latents of just those entries), then its window rows."""
    C, _ = ci.latent_rows_at(wl, b, sel, "cpu")
    key = np.zeros((1, len(sel), wl.d_idx), np.float32)
    codes, scales, _k, _s, _x, _ = O.append(C.reshape(1, -1, 512).numpy(), None, key, 1)
    return O.gather_rows(codes, scales, 0, np.arange(len(sel), dtype=np.int32), win_bits, wcap, t,
                         0, n_win)


def _peaky_q(rng, rows, cnt, H):
    """Attention queries (fp32) of one query whose rows are `rows` (selected
    entries first, then the window): heads 0-15 random at 16x the usual scale;
    16-31 aligned with a row three quarters into the selection; 32-47 aligned
    with a row an eighth into it; 48-55 aligned with one of the last window
    rows; 56-63 the usual N(0, 1/512)."""
    q = rng.normal(size=(H, 512)) / np.sqrt(512.0)
    q[:16] *= 16.0
    for h in range(16, 32):
        q[h] = rows[int(cnt * 0.75) + (h - 16) * (cnt // 80)] * (0.05 + 0.01 * (h - 16))
    for h in range(32, 48):
        q[h] = rows[cnt // 8 + (h - 32) * 3] * 0.08
    n_w = len(rows) - cnt
    for h in range(48, 56):
        q[h] = rows[cnt + n_w - 4 + (h % 4)] * 0.1
    return q


def _f32_of_bits(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("layout", ["one_split", "eight_splits"])
def test_attention_peaky_logits_rescale_and_split_merge(layout):
    H, n_win, wcap = 64, 128, 256
    if layout == "one_split":
        # 160 queries, one CTA each; three of them hold 2,048 selected rows (17
        # tiles in one CTA), the others a handful
        n_ent, nq = 2200, 160
        cnts = [16 + (i % 5) for i in range(nq)]
        big = [0, 77, 159]
        for i in big:
            cnts[i] = 2048
    else:
        # two queries split 16 ways: 8,000 + 128 rows (4 tiles per CTA) and 2,048 + 128
        n_ent, nq = 12000, 2
        cnts = [8000, 2048]
        big = [0, 1]
    wl = ci.Workload("t", nq, [n_ent] * nq, 0, 1, heads=H, seed=36)
    cache = build_gpu_cache(wl, DEV)
    rng = np.random.default_rng(36)
    k_max = max(cnts)
    idx = np.zeros((nq, k_max), np.int32)
    for i, c in enumerate(cnts):
        idx[i, :c] = np.sort(rng.choice(n_ent, c, replace=False))
    win = ci.window_rows(wl, nq, wcap, "cpu")
    t = n_ent - 1
    rows_of, q = {}, np.zeros((nq, H, 512))
    for i in range(nq):
        rows_of[i] = _sel_rows(wl, i, idx[i, :cnts[i]], bits16(win[i]), wcap, t, n_win)
        if i in big:
            q[i] = _peaky_q(rng, rows_of[i], cnts[i], H)
        else:
            q[i] = rng.normal(size=(H, 512)) / np.sqrt(512.0)
    qa = torch.from_numpy(q.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
    splits = _attn_splits(nq, k_max + n_win)
    assert splits == (1 if layout == "one_split" else 16)
    # the inputs drive the paths under test (checked on exact logits)
    rescaled_late, far_apart = False, False
    for i in big:
        lg = (rows_of[i] @ _f32_of_bits(bits16(qa[i])).T) * LOG2E       # [rows][H], log2 units
        parts = [p for p in _split_tiles(len(rows_of[i]), splits) if p]
        for tiles in parts:
            if len(tiles) > 1:
                first = lg[tiles[0][0]:tiles[0][1]].max(0)
                later = np.max([lg[a:b].max(0) for a, b in tiles[1:]], axis=0)
                rescaled_late |= bool((later > first + 8).any())
        if len(parts) > 1:
            sm = np.sort(np.array([lg[p[0][0]:p[-1][1]].max(0) for p in parts]), axis=0)
            far_apart |= bool(((sm[-1] - sm[-2]) > 20).any())
    assert rescaled_late
    assert far_apart or layout == "one_split"
    out = torch.full((nq, H, 512), float("nan"), device=DEV)
    lse = torch.full((nq, H), float("nan"), device=DEV)
    cnt = csa.new_counters()
    qs = csa.Queries(list(range(nq)), [t] * nq, 1, DEV)
    csa.sparse_attn(cache, qs, torch.from_numpy(idx).to(DEV),
                    torch.tensor(cnts, dtype=torch.int32, device=DEV), qa.to(DEV), win.to(DEV),
                    n_win, out, lse=lse, counters=cnt)
    torch.cuda.synchronize()
    assert _np(cnt).tolist() == [0, 0, 0, 0]
    go, gl = _np(out), _np(lse)
    for i in range(nq):
        ref, rlse = O.attention(bits16(qa[i]), rows_of[i], 1.0)
        err = rel_rows(go[i], ref)
        assert err.max() <= TOL, (i, int(err.argmax()), float(err.max()))
        assert np.abs(gl[i] - rlse).max() <= 1e-3 * max(1.0, np.abs(rlse).max()), i


# ---------------------------------------------------------------- layer top-k under heavy ties
@pytest.mark.parametrize("distinct", [1, 3, 400, 2000])
def test_layer_full_topk_with_few_distinct_scores(distinct):
    # A decode Full layer's top-k inside csa2_layer_step, with every entry's key
    # one of `distinct` integer vectors: scores tie by the tens of thousands
    # (1, 3: the threshold bin holds most of the row) or by the tens to
    # hundreds (400, 2000: ties at the k-th score spread over the row), and the
    # lowest positions must win among equal scores.
    n_ent, B, k = 40000, 2, 2048
    wl = ci.Workload("t", B, [n_ent] * B, 0, 1, exact=True, seed=41)
    cache = csa.Cache([n_ent + 8] * B, wl.d_idx, 1, DEV)
    g = torch.Generator().manual_seed(41)
    vecs = torch.randint(-8, 9, (distinct, wl.d_idx), generator=g).float()
    keys = []
    for b in range(B):
        C, _ = ci.latent_rows(wl, b, 0, n_ent, DEV)
        pick = torch.randint(0, distinct, (n_ent,), generator=g)
        keys.append(vecs[pick])
        csa.quantize_append(cache, C[None].contiguous(), None, keys[b][None].contiguous().to(DEV),
                            seq=b)
    qi, w, qa = ci.query_inputs(wl, B, "cpu")
    qs = csa.Queries(list(range(B)), [n_ent - 1] * B, 1, DEV)
    win = ci.window_rows(wl, B, 256, DEV)
    idx = torch.full((B, k), -1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros(B, dtype=torch.int32, device=DEV)
    out = torch.zeros(B, wl.heads, 512, device=DEV)
    counters = csa.new_counters()
    csa.Layer(csa.FULL, cache, qs, k=k, q=qa.to(DEV), win=win, n_win=wl.n_win, out=out, idx=idx,
              cnt=cnt, q_idx=qi.to(DEV), w=w.to(DEV), max_n=n_ent, counters=counters)()
    torch.cuda.synchronize()
    assert _np(counters).tolist() == [0, 0, 0, 0]
    for b in range(B):
        k8, ks = O.fp8_encode_rows(keys[b].numpy())
        sc = O.scores_full(k8, ks, qi[b].numpy(), w[b].numpy(), 0, n_ent)
        assert len(np.unique(sc)) <= distinct
        ref = O.topk(sc, k)
        assert int(cnt[b]) == k and np.array_equal(_np(idx[b]), ref), b
