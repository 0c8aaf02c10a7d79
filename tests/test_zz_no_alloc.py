"""csa2_topk_noalloc: top-k for callers that cannot allocate device memory
(for instance a plugin whose host program owns every device allocation, or a
serving loop that forbids allocating after start-up).  Its scratch is a fixed
array inside the library.  The test calls it through the C ABI and compares
it with csa2_topk, the entry point that takes a workspace, and with the
float64 oracle's top-k, on two calls in a row: the second call must not see
anything the first one left behind."""
import ctypes

import pytest
import numpy as np
import torch

import oracle as O
import sparse_attention_decode_step_gb300 as csa
from helpers import need_gpu

pytestmark = pytest.mark.gpu


def _noalloc():
    L = csa.lib()
    f = L.csa2_topk_noalloc
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f.argtypes = [vp, i64, vp, vp, i32, i32, i64, i32, vp, i64, vp, vp]
    f.restype = ctypes.c_int
    L.csa2_topk_noalloc_max_scratch.restype = ctypes.c_size_t
    return f, int(L.csa2_topk_noalloc_max_scratch())


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _case(seed, nq, n, dev):
    g = torch.Generator().manual_seed(seed)
    s = torch.randn(nq, n, generator=g)
    s[1::2] = torch.round(s[1::2] * 4) / 4            # many exact ties
    nv = torch.tensor([n - 3 * i for i in range(nq)], dtype=torch.int32)
    return s.to(dev), nv.to(dev)


def test_noalloc_topk_matches_workspace_topk_twice():
    need_gpu()
    dev = "cuda"
    fn, cap = _noalloc()
    assert cap == 4 << 20
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # one case above and one below 256K candidates: the two ways the selection
    # uses its scratch (chunked multi-CTA passes, one cluster per query)
    for seed, (nq, n, k) in enumerate([(3, 300000, 2048), (5, 16384, 512)]):
        scores, nv = _case(seed, nq, n, dev)
        assert csa.topk_workspace_size(nq, n) <= cap
        idx_a = torch.full((nq, k), -7, dtype=torch.int32, device=dev)
        cnt_a = torch.full((nq,), -7, dtype=torch.int32, device=dev)
        assert fn(_p(scores), n, _p(nv), None, 0, nq, n, k, _p(idx_a), k, _p(cnt_a), stream) == 0
        idx_b = torch.full((nq, k), -7, dtype=torch.int32, device=dev)
        cnt_b = torch.full((nq,), -7, dtype=torch.int32, device=dev)
        csa.topk(scores, nv, k, idx_b, cnt_b, max_n=n)
        torch.cuda.synchronize()
        # top-k indices are integers: the bar is identity
        assert torch.equal(cnt_a, cnt_b)
        assert torch.equal(idx_a, idx_b)
        assert int(cnt_a.min()) == min(k, n - 3 * (nq - 1))
        # and both equal the oracle's selection on the same fp32 scores
        s_h, nv_h = scores.cpu().numpy(), nv.cpu().numpy()
        ia, ca = idx_a.cpu().numpy(), cnt_a.cpu().numpy()
        for i in range(nq):
            ref = O.topk(s_h[i, :nv_h[i]], k)
            assert ca[i] == len(ref) and np.array_equal(ia[i, :ca[i]], ref), (seed, i)


def test_noalloc_topk_refuses_problems_beyond_its_scratch():
    need_gpu()
    fn, cap = _noalloc()
    p = ctypes.c_void_p(4096)
    nq, n = 512, 1 << 22
    assert csa.topk_workspace_size(nq, n) > cap
    assert fn(p, n, p, None, 0, nq, n, 2048, p, 2048, p, None) == -3   # CSA2_ERR_CAPACITY
