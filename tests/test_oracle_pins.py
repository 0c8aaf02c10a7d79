"""Pins of the float64 oracle against what the pages and mathematics fix.

Each check compares the oracle with something other than itself: the printed
figures (tests/golden/), exact rational arithmetic (fractions.Fraction), a
library routine (torch's float8 conversion, softmax and scaled-dot-product
attention, numpy GEMV), or brute force on tiny inputs.  They run on the CPU.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from conftest import golden, read_constants

PAGES = read_constants()


# --------------------------------------------------------------- formats
def _torch_e4m3_table():
    b = torch.arange(256, dtype=torch.uint8)
    return b.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e2m1_table_matches_golden():
    # [Notes] section 4: E2M1 elements
    rows = [l.split() for l in open(golden("e2m1_values.txt")) if l.strip() and not l.startswith("#")]
    for code, val in rows:
        got = O.e2m1_value(int(code))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code


def test_e4m3_decode_matches_library():
    tab = _torch_e4m3_table()
    for b in range(256):
        ours = O.e4m3_value(b)
        if math.isnan(tab[b]):
            assert math.isnan(ours), b
        else:
            assert ours == tab[b], b


def test_e4m3_constants():
    pos = [O.e4m3_value(b) for b in range(1, 0x7F)]
    assert len(pos) == 126 and all(np.diff(pos) > 0)
    assert max(pos) == PAGES["e4m3_max"]            # 448
    assert min(pos) == 2.0 ** -9
    assert O.e4m3_value(0x38) == 1.0


def test_fp4_range_is_paper_figure():
    # [Notes] section 4: representable range 448 x 6 = 2688
    top = max(O.e2m1_value(c) for c in range(16)) * max(O.e4m3_value(b) for b in range(0x7F))
    assert top == PAGES["fp4_range"] == PAGES["e4m3_max"] * PAGES["e2m1_max"]


def test_e4m3_nearest_matches_library_rne():
    tab = _torch_e4m3_table()
    pos = np.array([tab[b] for b in range(0x7F)])
    mids = (pos[:-1] + pos[1:]) / 2
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        rng.uniform(-448, 448, 4000), rng.normal(0, 1, 2000), rng.normal(0, 1e-2, 1000),
        mids, -mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)).astype(np.float64),
        np.nextafter(mids.astype(np.float32), np.float32(0)).astype(np.float64),
    ]).astype(np.float32)
    lib = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy().astype(int)
    for x, lb in zip(xs, lib):
        ours = O.e4m3_nearest(float(x))
        if lb & 0x7F == 0:
            lb = 0                                    # canonical zero byte
        assert ours == lb, (x, ours, lb)


def test_fp8_pow2_scale_definition():
    for amax in [0.0, 1e-30, 1e-3, 0.5, 1.0, 447.9, 448.0, 448.0001, 1000.0, 3.4e38]:
        s = O.fp8_pow2_scale(amax)
        if amax == 0:
            assert s == 1.0
            continue
        e = math.frexp(s)[1] - 1
        assert s == 2.0 ** e
        assert Fraction(448) * Fraction(s) >= Fraction(amax)
        assert Fraction(448) * Fraction(s) / 2 < Fraction(amax)


# --------------------------------------------------------------- FP4 encode
_E2M1 = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
         Fraction(4), Fraction(6)]


def _exact_scale_byte(amax):
    tab = _torch_e4m3_table()
    for b in range(1, 0x7F):
        if 6 * Fraction(tab[b]) >= Fraction(amax):
            return b
    return 0x7E


def _exact_code(x, s):
    ax = abs(Fraction(x))
    s = Fraction(s)
    d = [abs(ax - v * s) for v in _E2M1]
    best = min(range(8), key=lambda i: (d[i], i % 2))   # nearest, ties to the even index
    if best == 0:
        return 0
    return (8 | best) if x < 0 else best


def _check_group(vals):
    x = np.zeros(512)
    x[:16] = vals
    codes, scales, nsat = O.fp4_encode_entry(x)
    amax = float(np.max(np.abs(vals)))
    want_sb = 0 if amax == 0 else _exact_scale_byte(amax)
    assert scales[0] == want_sb, (vals, scales[0], want_sb)
    s = O.e4m3_value(want_sb)
    for c in range(16):
        nib = (codes[c // 2] >> (4 * (c % 2))) & 15
        want = 0 if want_sb == 0 else _exact_code(vals[c], s)
        assert nib == want, (c, vals[c], s, nib, want)
    return nsat


def test_fp4_encode_random_groups_exact():
    rng = np.random.default_rng(11)
    for _ in range(300):
        scale = 10.0 ** rng.uniform(-3, 2.5)
        _check_group(rng.normal(0, scale, 16).astype(np.float32).astype(np.float64))


def test_fp4_encode_ties_and_neighbours():
    # every E2M1 midpoint times a scale, and one float32 ulp either side of it
    mids = [Fraction(1, 4), Fraction(3, 4), Fraction(5, 4), Fraction(7, 4), Fraction(5, 2),
            Fraction(7, 2), Fraction(5)]
    rng = np.random.default_rng(3)
    for sb in [0x08, 0x20, 0x33, 0x38, 0x3D, 0x48, 0x55, 0x7E]:
        s = O.e4m3_value(sb)
        for mid in mids:
            m = float(mid * Fraction(s))
            assert Fraction(np.float32(m).item()) == mid * Fraction(s)   # exact in fp32
            for v in [m, float(np.nextafter(np.float32(m), np.float32(np.inf))),
                      float(np.nextafter(np.float32(m), np.float32(0)))]:
                vals = rng.uniform(-1, 1, 16) * 0.1 * s
                vals[0] = 6 * s                       # pins the scale to byte sb
                vals[1] = v
                vals[2] = -v
                _check_group(vals)


def test_fp4_saturation_and_zero():
    assert _check_group(np.full(16, 2688.0)) == 0
    assert _check_group(np.array([2688.0 * (1 + 2 ** -20)] + [0.0] * 15)) == 1
    assert _check_group(np.zeros(16)) == 0
    x = np.zeros(16)
    x[3] = -0.0
    x[5] = -1e-3
    x[6] = 1.0
    _check_group(x)


def test_fp4_roundtrip_of_representable_values():
    rng = np.random.default_rng(5)
    for _ in range(100):
        sb = int(rng.integers(1, 0x7F))
        s = O.e4m3_value(sb)
        idx = rng.integers(0, 8, 16)
        sign = rng.choice([-1, 1], 16)
        vals = sign * np.array([float(_E2M1[i]) for i in idx]) * s
        vals[0] = 6 * s
        codes, scales, _ = O.fp4_encode_entry(np.pad(vals, (0, 496)))
        dec = O.fp4_decode_entry(codes, scales)[:16]
        assert np.array_equal(dec, vals)


def test_fp4_granularity_and_bytes_per_entry():
    codes, scales, _ = O.fp4_encode_entry(np.ones(512))
    assert codes.nbytes == 256 and scales.nbytes == 32
    assert scales.nbytes == PAGES["latent_width"] / PAGES["scale_group"]
    assert (codes.nbytes + scales.nbytes) * 8 / 512 == 4.5


def test_norm_bound_never_saturates():
    # [Notes] section 4: RMSNorm bounds ||v|| by sqrt(512), RoPE is orthogonal, so
    # max |v_i| <= sqrt(512) ~ 22.6; with range 2688 no group saturates and the
    # scale never exceeds the smallest E4M3 >= 22.63 / 6, which is 4.0.
    bound = math.sqrt(512)
    assert abs(bound - PAGES["latent_bound"]) < 0.05
    rng = np.random.default_rng(9)
    cases = []
    for i in range(0, 512, 37):
        x = np.zeros(512)
        x[i] = bound * (1 if i % 2 else -1)          # one-hot spike at the bound
        cases.append(x)
    for _ in range(40):
        v = rng.normal(size=512)
        v *= bound / np.linalg.norm(v)
        q, _r = np.linalg.qr(rng.normal(size=(512, 512)))
        cases.append(q @ v)                           # orthogonal map keeps the norm
    for x in cases:
        assert np.linalg.norm(x) <= bound * (1 + 1e-12)
        codes, scales, nsat = O.fp4_encode_entry(x)
        assert nsat == 0
        assert max(O.e4m3_value(int(s)) for s in scales) <= 4.0


# --------------------------------------------------------------- compression
def test_compression_special_cases_and_softmax_library():
    rng = np.random.default_rng(13)
    for m in (1, 2, 4):
        C = rng.normal(size=(m, 512)).astype(np.float32)
        Z = rng.normal(size=(m, 512)).astype(np.float32)
        got = O.compress_block(C, Z, m)
        Ct, Zt = torch.from_numpy(C).double(), torch.from_numpy(Z).double()
        want = (torch.softmax(Zt, dim=0) * Ct).sum(0).numpy()
        assert np.allclose(got, want, rtol=1e-13, atol=1e-15)
        assert np.all(np.abs(got) <= np.abs(C).max(0) + 1e-12)   # convex combination
    C = rng.normal(size=(1, 512)).astype(np.float32)
    assert np.array_equal(O.compress_block(C, None, 1), C[0].astype(np.float64))
    C = rng.normal(size=(2, 512)).astype(np.float32)
    Zeq = np.tile(rng.normal(size=(1, 512)).astype(np.float32), (2, 1))
    assert np.allclose(O.compress_block(C, Zeq, 2), C.astype(np.float64).mean(0), rtol=0, atol=1e-15)
    Zgap = np.zeros((2, 512), np.float32)
    Zgap[1] = 250.0                                   # exp(-250) vanishes against 1
    assert np.array_equal(O.compress_block(C, Zgap, 2), C[1].astype(np.float64))


def test_append_batch_layout():
    rng = np.random.default_rng(17)
    B, n_tok, m, d = 2, 6, 2, 64
    C = rng.normal(size=(B, n_tok, 512)).astype(np.float32)
    Z = rng.normal(size=(B, n_tok, 512)).astype(np.float32)
    key = rng.normal(size=(B, n_tok // m, d)).astype(np.float32)
    codes, scales, kidx, ksc, x, nsat = O.append(C, Z, key, m)
    assert codes.shape == (6, 256) and kidx.shape == (6, 64) and nsat == 0
    for b in range(B):
        for e in range(n_tok // m):
            r = b * (n_tok // m) + e
            assert np.allclose(x[r], O.compress_block(C[b, e * m:(e + 1) * m], Z[b, e * m:(e + 1) * m], m))
            c2, s2, _ = O.fp4_encode_entry(x[r])
            assert np.array_equal(c2, codes[r]) and np.array_equal(s2, scales[r])
            k8, ks = O.fp8_encode_rows(key[b, e][None])
            assert np.array_equal(k8[0], kidx[r]) and ks[0] == ksc[r]


# --------------------------------------------------------------- projected indexer key
def _bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def _bf16_values(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def _dequant_entries(codes, scales):
    # decode with the golden E2M1 table and the library's E4M3 decode
    e2m1 = {int(c): float(v) for c, v in (l.split() for l in open(golden("e2m1_values.txt"))
                                          if l.strip() and not l.startswith("#"))}
    nib = np.stack([codes & 15, codes >> 4], -1).reshape(codes.shape[0], 512)
    vals = np.vectorize(e2m1.get)(nib).astype(np.float64)
    return vals * np.repeat(_torch_e4m3_table()[scales.astype(np.int64)], 16, axis=1)


def test_append_project_is_stored_entry_times_w():
    # key = (dequantised stored entry) @ W_IK, then the FP8 encoding of a given key
    rng = np.random.default_rng(41)
    for m, d in ((1, 128), (2, 64)):
        C = rng.normal(size=(2, 4 * m, 512)).astype(np.float32)
        Z = rng.normal(size=(2, 4 * m, 512)).astype(np.float32)
        wbits = _bf16_bits(rng.normal(size=(512, d)) / 16)
        codes, scales, kidx, ksc, k, nsat = O.append_project(C, Z, wbits, m)
        c2, s2, _k, _s, _x, _ = O.append(C, Z, np.zeros((2, 4, d), np.float32), m)
        assert np.array_equal(codes, c2) and np.array_equal(scales, s2) and nsat == 0
        want = _dequant_entries(codes, scales) @ _bf16_values(wbits)      # numpy matmul
        assert np.allclose(k, want, rtol=1e-12, atol=1e-12)
        # FP8 step: the library's round-to-nearest-even E4M3 of k / scale
        lib8 = torch.from_numpy(k / ksc[:, None].astype(np.float64)).to(
            torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(kidx, lib8)
        assert all(ks == O.fp8_pow2_scale(np.abs(kk).max()) for kk, ks in zip(k, ksc))


def test_append_project_identity_rows_give_the_entry():
    # W = [I; 0]: the key is the first d channels of the stored entry (pins the
    # orientation: row c of W_IK multiplies latent channel c)
    rng = np.random.default_rng(42)
    C = rng.normal(size=(1, 3, 512)).astype(np.float32)
    w = np.zeros((512, 128), np.float32)
    w[np.arange(128), np.arange(128)] = 1.0
    codes, scales, _kidx, _ksc, k, _ = O.append_project(C, None, _bf16_bits(w), 1)
    assert np.array_equal(k, _dequant_entries(codes, scales)[:, :128])


def test_append_project_exact_inputs_are_exact():
    # integer latents in [-6, 6] with a 6 in every 16-channel group: every scale
    # is 1.0, stored values are multiples of 1/2, and with W_IK entries k / 64
    # every product and partial sum is a multiple of 1/128 below 2^12 -- exact
    # in fp32 in any order, so a fp32 kernel and this fp64 oracle agree bit for bit
    rng = np.random.default_rng(43)
    C = rng.integers(-6, 7, size=(1, 5, 512)).astype(np.float32)
    C[..., ::16] = 6.0
    w = rng.integers(-64, 65, size=(512, 128)) / 64.0
    codes, scales, kidx, ksc, k, _ = O.append_project(C, None, _bf16_bits(w), 1)
    assert (scales == 0x38).all()
    assert np.array_equal(k * 128, np.round(k * 128)) and np.abs(k).max() < 4096
    assert np.array_equal(k.astype(np.float32).astype(np.float64), k)


# --------------------------------------------------------------- scores
def _dequant_fp8(b, s):
    return _torch_e4m3_table()[b.astype(np.int64)] * s[..., None]


def test_scores_reduce_to_relu_gemv():
    # one indexer head with unit weight: score = ReLU(K q), a plain GEMV
    rng = np.random.default_rng(19)
    n, d = 300, 128
    key = rng.normal(size=(n, d)).astype(np.float32)
    k8, ks = O.fp8_encode_rows(key)
    q = rng.normal(size=(1, d)).astype(np.float32)
    q8, qs = O.fp8_encode_rows(q)
    got = O.scores_full(k8, ks, q, np.ones(1, np.float32), 0, n)
    want = np.maximum(_dequant_fp8(k8, ks) @ _dequant_fp8(q8, qs)[0], 0.0)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_scores_multi_head_formula():
    rng = np.random.default_rng(23)
    n, d, h = 200, 64, 4
    key = rng.normal(size=(n, d)).astype(np.float32)
    k8, ks = O.fp8_encode_rows(key)
    q = rng.normal(size=(h, d)).astype(np.float32)
    w = rng.uniform(size=h).astype(np.float32)
    w[1] = -0.5                                       # negative weights allowed
    q8, qs = O.fp8_encode_rows(q)
    got = O.scores_full(k8, ks, q, w, 0, n)
    dots = _dequant_fp8(k8, ks) @ _dequant_fp8(q8, qs).T       # [n][h]
    want = (np.maximum(dots, 0) * w.astype(np.float64)).sum(1)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    rows = np.array([5, 7, 199, 0], np.int64)
    assert np.array_equal(O.scores_at(k8, ks, q, w, rows), got[rows])


def test_scores_exact_integer_mode():
    rng = np.random.default_rng(29)
    n, d, h = 256, 128, 8
    key = rng.integers(-8, 9, (n, d)).astype(np.float32)
    q = rng.integers(-8, 9, (h, d)).astype(np.float32)
    w = (rng.integers(0, 17, h) / 16).astype(np.float32)
    k8, ks = O.fp8_encode_rows(key)
    got = O.scores_full(k8, ks, q, w, 0, n)
    want = (np.maximum(key.astype(np.int64) @ q.astype(np.int64).T, 0) * w.astype(np.float64)).sum(1)
    assert np.array_equal(got, want)


# --------------------------------------------------------------- top-k
def _brute_topk(scores, k, pos=None):
    pos = np.arange(len(scores)) if pos is None else np.asarray(pos)
    order = np.lexsort((pos, -np.asarray(scores, np.float64)))
    return np.sort(pos[order[:k]])


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(31)
    for trial in range(200):
        n = int(rng.integers(1, 300))
        k = int(rng.integers(1, 64))
        sc = rng.integers(-5, 6, n).astype(np.float64) * 0.5   # many exact ties
        if trial % 3 == 0:
            sc[rng.integers(0, n, 3)] = -0.0
        assert np.array_equal(O.topk(sc, k), _brute_topk(sc, k))


def test_topk_fewer_candidates_than_k_returns_all():
    sc = np.array([3.0, -1.0, 2.0])
    assert np.array_equal(O.topk(sc, 10), [0, 1, 2])
    assert len(O.topk(np.zeros(0), 4)) == 0


def test_topk_with_position_map():
    rng = np.random.default_rng(37)
    pos = np.sort(rng.choice(10000, 200, replace=False)).astype(np.int32)
    sc = rng.integers(0, 4, 200).astype(np.float64)
    assert np.array_equal(O.topk(sc, 50, pos), _brute_topk(sc, 50, pos))


# --------------------------------------------------------------- pool
def test_blockmax_matches_reshape_max():
    rng = np.random.default_rng(41)
    for n in (1, 7, 8, 9, 1000, 1003):
        sc = rng.normal(size=n)
        pad = np.full((-n) % 8, -np.inf)
        assert np.array_equal(O.blockmax(sc), np.concatenate([sc, pad]).reshape(-1, 8).max(1))


def test_pool_small_context_is_whole_context():
    # [Notes] section 3: a constant-size pool holds nearly all of a short context
    rng = np.random.default_rng(43)
    for n in (5, 4096, 16384, 16381):
        blk, pn = O.pool(rng.normal(size=n), 2048)
        assert pn == n and np.array_equal(blk, np.arange((n + 7) // 8))


def test_pool_size_at_1m_is_paper_figure():
    # [Notes] section 3: 2,048 x 8 = 16,384 positions; 1.6% of a 1M context
    n = 1 << 20
    sc = np.random.default_rng(47).normal(size=n)
    blk, pn = O.pool(sc, int(PAGES["pool_blocks"]))
    assert len(blk) == PAGES["pool_blocks"] and pn == PAGES["pool_positions"]
    assert round(100 * pn / n, 1) == PAGES["pool_fraction_1m_pct"]
    assert np.all(np.diff(blk) > 0)
    bm = O.blockmax(sc)
    assert np.array_equal(blk, np.sort(np.lexsort((np.arange(len(bm)), -bm))[:2048]))


def test_pool_partial_last_block():
    # the block holding the newest entries may be partial: only its visible
    # entries score it and count towards the pool
    rng = np.random.default_rng(79)
    n = 8 * 3000 + 3
    sc = rng.normal(size=n)
    sc[-3:] = 50.0                                    # make the partial block a winner
    blk, pn = O.pool(sc, 2048)
    pad = np.concatenate([sc, np.full(5, -np.inf)]).reshape(-1, 8).max(1)
    assert np.array_equal(blk, np.sort(np.lexsort((np.arange(len(pad)), -pad))[:2048]))
    assert blk[-1] == n // 8 and pn == 8 * 2047 + 3


def _cache_from_latents(rng, n, d_idx, exact=False):
    C = rng.normal(size=(1, n, 512)).astype(np.float32)
    if exact:
        key = rng.integers(-8, 9, (1, n, d_idx)).astype(np.float32)
    else:
        key = rng.normal(size=(1, n, d_idx)).astype(np.float32)
    codes, scales, kidx, ksc, _x, _ = O.append(C, None, key, 1)
    return codes, scales, kidx, ksc


def test_reindex_with_full_query_reproduces_full_topk():
    # Every block holding a top-k entry has block max >= the k-th score, so for
    # k <= 2048 all such blocks are in the pool and rescoring the pool with the
    # Full layer's own query returns the same k positions.
    rng = np.random.default_rng(53)
    n, d_idx, h_idx = 40000, 64, 4
    codes, scales, kidx, ksc = _cache_from_latents(rng, n, d_idx)
    q_idx = rng.normal(size=(1, h_idx, d_idx)).astype(np.float32)
    w = rng.uniform(size=(1, h_idx)).astype(np.float32)
    qa = torch.randn(1, 16, 512).mul(512 ** -0.5).to(torch.bfloat16).view(torch.int16).numpy()
    common = dict(codes=codes, scales=scales, kidx=kidx, kscale=ksc, seq_base=[0], m=1,
                  q_seq=[0], q_pos=[n - 1], H=16, q_attn=qa, win=None, wcap=1, n_win=0,
                  sm_scale=1.0, q_idx=q_idx, w=w)
    for k in (64, 512, 2048):
        full = O.layer(O.FULL, k=k, build_pool=True, **common)
        re = O.layer(O.REINDEX, k=k, pool_blk=full["pool_blk"], pool_n=full["pool_n"], **common)
        assert full["pool_n"][0] == 16384
        assert np.array_equal(full["idx"], re["idx"]) and full["cnt"][0] == re["cnt"][0] == k
        assert np.allclose(full["out"], re["out"], rtol=0, atol=0)


# --------------------------------------------------------------- attention
def _sdpa(q_bits, rows, sm_scale):
    q = torch.from_numpy(q_bits).view(torch.bfloat16).double()[None]        # [1][H][512]
    kv = torch.from_numpy(rows).double()[None, None].expand(1, q.shape[1], -1, -1)
    out = torch.nn.functional.scaled_dot_product_attention(q, kv, kv, scale=sm_scale)
    return out[0].numpy()


def test_attention_matches_library_sdpa():
    rng = np.random.default_rng(59)
    for H, n, sm in ((16, 37, 1.0), (64, 300, 0.7)):
        rows = rng.normal(size=(n, 512))
        q = torch.from_numpy(rng.normal(size=(H, 512)) / 8).to(torch.bfloat16).view(torch.int16).numpy()
        out, lse = O.attention(q, rows, sm)
        assert np.allclose(out, _sdpa(q, rows, sm), rtol=1e-10, atol=1e-12)
        qd = torch.from_numpy(q).view(torch.bfloat16).double().numpy()
        assert np.allclose(lse, np.log(np.exp(sm * qd @ rows.T).sum(1)), rtol=1e-12)


def test_window_truncation_formula():
    # [Notes] section 5: the window of position i is [max(s, i - n_win + 1), i]
    rng = np.random.default_rng(61)
    wcap = 256
    win = torch.from_numpy(rng.normal(size=(wcap, 512))).to(torch.bfloat16).view(torch.int16).numpy()
    codes = np.zeros((1, 256), np.uint8)
    scales = np.zeros((1, 32), np.uint8)
    for t, s, n_win in ((500, 0, 128), (500, 450, 128), (10, 0, 128), (300, 0, 1), (0, 0, 128)):
        rows = O.gather_rows(codes, scales, 0, [], win, wcap, t, s, n_win)
        lo = max(s, t - n_win + 1, 0)
        want = [win[p % wcap] for p in range(lo, t + 1)]
        want = torch.from_numpy(np.array(want)).view(torch.bfloat16).double().numpy()
        assert rows.shape[0] == t - lo + 1 and np.array_equal(rows, want)


def test_layer_with_k_at_least_context_is_dense_attention():
    rng = np.random.default_rng(67)
    n, d_idx, h_idx, H, wcap, n_win = 300, 64, 4, 16, 512, 128
    codes, scales, kidx, ksc = _cache_from_latents(rng, n, d_idx)
    q_idx = rng.normal(size=(1, h_idx, d_idx)).astype(np.float32)
    w = rng.uniform(size=(1, h_idx)).astype(np.float32)
    qa = torch.from_numpy(rng.normal(size=(1, H, 512)) / 22.6).to(torch.bfloat16).view(torch.int16).numpy()
    win = torch.from_numpy(rng.normal(size=(1, wcap, 512))).to(torch.bfloat16).view(torch.int16).numpy()
    t = n - 1
    res = O.layer(O.FULL, codes=codes, scales=scales, kidx=kidx, kscale=ksc, seq_base=[0], m=1,
                  q_seq=[0], q_pos=[t], k=512, H=H, q_attn=qa, win=win, wcap=wcap, n_win=n_win,
                  sm_scale=0.9, q_idx=q_idx, w=w)
    assert res["cnt"][0] == n and np.array_equal(res["idx"][0, :n], np.arange(n))
    rows = np.concatenate([O.fp4_decode_rows(codes, scales),
                           torch.from_numpy(win[0, t - n_win + 1:t + 1]).view(torch.bfloat16).double().numpy()])
    assert np.allclose(res["out"][0], _sdpa(qa[0], rows, 0.9), rtol=1e-10, atol=1e-12)
    # causality: entries past the query's visible range never matter
    codes2, scales2 = codes.copy(), scales.copy()
    res2 = O.layer(O.FULL, codes=np.concatenate([codes2, rng.integers(0, 256, (50, 256), dtype=np.uint8)]),
                   scales=np.concatenate([scales2, rng.integers(0, 0x7E, (50, 32), dtype=np.uint8)]),
                   kidx=np.concatenate([kidx, rng.integers(0, 0x7E, (50, d_idx), dtype=np.uint8)]),
                   kscale=np.concatenate([ksc, np.ones(50, np.float32)]), seq_base=[0], m=1,
                   q_seq=[0], q_pos=[t], k=512, H=H, q_attn=qa, win=win, wcap=wcap, n_win=n_win,
                   sm_scale=0.9, q_idx=q_idx, w=w)
    assert np.array_equal(res["out"], res2["out"])


def test_reuse_mode_needs_no_indexer_state():
    # [Deep read] section 03: Reuse takes the index list and skips the indexer
    rng = np.random.default_rng(71)
    n, H = 64, 16
    codes, scales, _k, _s = _cache_from_latents(rng, n, 64)
    qa = torch.from_numpy(rng.normal(size=(1, H, 512)) / 22.6).to(torch.bfloat16).view(torch.int16).numpy()
    idx = np.array([[3, 9, 40, 63]], np.int32)
    res = O.layer(O.REUSE, codes=codes, scales=scales, kidx=None, kscale=None, seq_base=[0], m=1,
                  q_seq=[0], q_pos=[n - 1], k=4, H=H, q_attn=qa, win=None, wcap=1, n_win=0,
                  sm_scale=1.0, idx=idx, cnt=[4])
    rows = O.fp4_decode_rows(codes[idx[0]], scales[idx[0]])
    assert np.allclose(res["out"][0], _sdpa(qa[0], rows, 1.0), rtol=1e-10, atol=1e-12)


def test_m2_visibility_counts_complete_blocks():
    # a query at token t sees floor((t + 1) / m) compressed entries
    rng = np.random.default_rng(73)
    codes, scales, kidx, ksc = _cache_from_latents(rng, 40, 64)
    qa = np.zeros((1, 16, 512), np.int16)
    for t in (0, 1, 2, 7, 8, 79):
        res = O.layer(O.FULL, codes=codes, scales=scales, kidx=kidx, kscale=ksc, seq_base=[0], m=2,
                      q_seq=[0], q_pos=[t], k=1000, H=16, q_attn=qa, win=None, wcap=1, n_win=0,
                      sm_scale=1.0, q_idx=np.ones((1, 4, 64), np.float32), w=np.ones((1, 4), np.float32))
        assert res["cnt"][0] == (t + 1) // 2


# --------------------------------------------------------------- accounting
def test_kv_bytes_per_token_accounting():
    # [Notes] intro: 890 B/token of global KV.  Encoder: 3 Full layers each own a
    # cache at m = 2 (0.5 entry/token each); decoder: one cache at m = 1.  An
    # entry is 288 B of FP4 latent + d_I key bytes + a 4-byte key scale; at
    # d_I = 64 this gives exactly the printed figure (a reading, not a claim).
    codes, scales, _ = O.fp4_encode_entry(np.ones(512))
    entries_per_token = 3 * (1 / 2) + 1 * 1
    per_entry = codes.nbytes + scales.nbytes + 64 + 4
    assert entries_per_token * per_entry == PAGES["global_kv_bytes_per_token"]
