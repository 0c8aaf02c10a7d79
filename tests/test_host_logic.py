"""Host-side logic that needs no GPU: the static layer schedule, and the
replica (multi-process) timing reduction bench.py uses for N > 1, run as two
gloo ranks on the CPU."""
import os

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT, read_constants
from sparse_attention_decode_step_gb300 import schedule as S

PAGES = read_constants()


def test_indexer_count_matches_pages():
    # [Notes] section 2: 3 indexers in the encoder, 5 in the decoder, 40 layers
    enc, dec = S.encoder_schedule(), S.decoder_schedule()
    assert len(enc) == 20 and len(dec) == 20 and len(enc) + len(dec) == PAGES["layers_total"]
    assert len(S.indexer_layers(enc)) == PAGES["indexers_encoder"]
    assert len(S.indexer_layers(dec)) == PAGES["indexers_decoder"]


def test_decoder_blocks_and_reuse_sources():
    dec = S.decoder_schedule()
    modes = [p.mode for p in dec]
    assert modes[:4] == [S.FULL, S.REUSE, S.REUSE, S.REUSE]
    for b in range(1, 5):
        assert modes[4 * b:4 * b + 4] == [S.REINDEX, S.REUSE, S.REUSE, S.REUSE]
    for p in dec:
        if p.mode == S.REUSE:
            src = dec[p.source - 1]
            assert src.mode in (S.FULL, S.REINDEX) and src.layer < p.layer
            assert all(q.mode == S.REUSE for q in dec[src.layer:p.layer - 1])   # nearest one
    assert [p.builds_pool for p in dec].count(True) == 1 and dec[0].builds_pool
    assert {p.m for p in dec} == {1}


def test_encoder_blocks():
    enc = S.encoder_schedule()
    assert [p.mode for p in enc[:2]] == [S.SWA, S.SWA]
    for b in range(3):
        blk = enc[2 + 6 * b:8 + 6 * b]
        assert [p.mode for p in blk] == [S.FULL] + [S.REUSE] * 5
        assert all(p.m == 2 and p.cache == b for p in blk)


def test_encoder_csa2_layers_for_the_chunk_driver():
    # the 18 layers EncoderChunk runs: blocks of 1 Full + 5 Reuse, block b on cache b,
    # every Reuse layer fed by its own block's Full layer
    plan = S.encoder_csa2_layers()
    assert [p.layer for p in plan] == list(range(3, 21))
    for b in range(3):
        blk = plan[6 * b:6 * b + 6]
        assert [p.mode for p in blk] == [S.FULL] + [S.REUSE] * 5
        assert {p.cache for p in blk} == {b} and {p.m for p in blk} == {2}
        assert all(p.source == blk[0].layer for p in blk[1:])


def test_entries_per_token_and_kv_accounting():
    # three m = 2 encoder caches + one m = 1 decoder cache = 2.5 entries per token;
    # at 288 + 64 + 4 B per entry that is the pages' 890 B/token
    ept = S.entries_per_token()
    assert ept == 2.5
    assert ept * (288 + 64 + 4) == PAGES["global_kv_bytes_per_token"]


def _replica_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = 0.010 * (rank + 1)              # rank 1 is the slower replica
    t = bench.job_time(local, world, "cpu")
    v = bench.job_value(32 * 10, world, t)
    q.put((rank, t, v))
    dist.barrier()
    dist.destroy_process_group()


def test_replica_timing_reduction_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29600 + os.getpid() % 1000
    procs = [ctx.Process(target=_replica_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = {r: (t, v) for r, t, v in (q.get(timeout=180) for _ in procs)}
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time; throughput counts both replicas' queries
    assert got[0] == got[1] == (0.020, 2 * 320 / 0.020)
