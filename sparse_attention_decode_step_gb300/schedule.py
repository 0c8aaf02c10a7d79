"""Static CSA2 layer schedules and a decoder-step driver over the C ABI.

[Notes] section 2: the encoder's layers 1-2 are pure sliding-window
attention and layers 3-20 are three 6-layer CSA2 blocks of 1 Full + 5 Reuse
at m = 2; the decoder is five 4-layer blocks at m = 1, the first 1 Full +
3 Reuse, the other four 1 Reindex + 3 Reuse -- 3 + 5 indexers in 40 layers.
[Deep read] section 03: Reindex reuses the Full layer's main KV and indexer
K with its own indexer query; Reuse takes the index list of the nearest
preceding Full or Reindex layer and computes only its own query, window KV
and attention.  The decoder's first Full layer also builds the candidate
pool ([Notes] section 3) that the Reindex layers search.
"""
from __future__ import annotations

from dataclasses import dataclass

SWA, FULL, REINDEX, REUSE = "swa", "full", "reindex", "reuse"


@dataclass(frozen=True)
class LayerPlan:
    layer: int          # 1-based layer number within its stack
    mode: str
    m: int              # block-compression factor of the cache it reads (0 for SWA)
    cache: int          # index of the main-KV cache it reads (-1 for SWA)
    source: int         # layer whose index list a Reuse layer takes (-1 otherwise)
    builds_pool: bool


def encoder_schedule():
    plan = [LayerPlan(1, SWA, 0, -1, -1, False), LayerPlan(2, SWA, 0, -1, -1, False)]
    for blk in range(3):
        first = 3 + 6 * blk
        plan.append(LayerPlan(first, FULL, 2, blk, -1, False))
        for j in range(1, 6):
            plan.append(LayerPlan(first + j, REUSE, 2, blk, first, False))
    return plan


def decoder_schedule():
    plan = []
    for blk in range(5):
        first = 1 + 4 * blk
        if blk == 0:
            plan.append(LayerPlan(first, FULL, 1, 0, -1, True))
        else:
            plan.append(LayerPlan(first, REINDEX, 1, 0, -1, False))
        for j in range(1, 4):
            plan.append(LayerPlan(first + j, REUSE, 1, 0, first, False))
    return plan


def indexer_layers(plan):
    return [p.layer for p in plan if p.mode in (FULL, REINDEX)]


def entries_per_token(enc=None, dec=None):
    """Main-KV entries stored per token: one cache per Full layer, 1/m entries each."""
    enc = encoder_schedule() if enc is None else enc
    dec = decoder_schedule() if dec is None else dec
    return sum(1.0 / p.m for p in enc + dec if p.mode == FULL)


class DecoderStep:
    """Runs one decode step of the 20-layer decoder through csa2_layer_step.

    per_layer[l] holds layer l+1's own inputs: q_idx, w (Full/Reindex only),
    q (attention queries), win (window KV ring), out, optional lse.  Reuse
    layers read the index list of their source layer; the Full layer builds
    the pool that the Reindex layers score.  One workspace serves every layer
    in turn."""

    def __init__(self, csa, cache, qs, per_layer, *, k, n_win, max_n, pool_blocks=2048,
                 sm_scale=1.0, counters=None):
        import torch
        self.plan = decoder_schedule()
        dev = per_layer[0]["q"].device
        nq = qs.nq
        self.pool_blk = torch.zeros(nq, pool_blocks, dtype=torch.int32, device=dev)
        self.pool_n = torch.zeros(nq, dtype=torch.int32, device=dev)
        self.idx = {p.layer: torch.zeros(nq, k, dtype=torch.int32, device=dev)
                    for p in self.plan if p.mode in (FULL, REINDEX)}
        self.cnt = {p.layer: torch.zeros(nq, dtype=torch.int32, device=dev)
                    for p in self.plan if p.mode in (FULL, REINDEX)}
        modes = {FULL: csa.FULL, REINDEX: csa.REINDEX, REUSE: csa.REUSE}
        ws = None
        self.layers = []
        for p in self.plan:
            L = per_layer[p.layer - 1]
            src = p.layer if p.mode != REUSE else p.source
            indexer = p.mode != REUSE
            layer = csa.Layer(modes[p.mode], cache, qs, k=k, q=L["q"], win=L["win"], n_win=n_win,
                              out=L["out"], idx=self.idx[src], cnt=self.cnt[src],
                              q_idx=L.get("q_idx") if indexer else None,
                              w=L.get("w") if indexer else None, max_n=max_n,
                              build_pool=p.builds_pool, pool_blocks=pool_blocks,
                              pool_blk=self.pool_blk, pool_n=self.pool_n, lse=L.get("lse"),
                              sm_scale=sm_scale, counters=counters, ws=ws)
            ws = layer.ws
            self.layers.append(layer)

    def __call__(self):
        for layer in self.layers:
            layer()


def encoder_csa2_layers():
    """The encoder's CSA2 layers (3..20) in order: three blocks of 1 Full +
    5 Reuse at m = 2, block b reading main-KV cache b."""
    return [p for p in encoder_schedule() if p.mode != SWA]


class EncoderChunk:
    """Runs the encoder's 18 CSA2 layers over one chunk of prompt queries
    through csa2_layer_step.

    [Notes] section 2: each Full layer keeps its own compressed cache (here
    caches[0..2], m = 2, one per block, the chunk's own tokens already
    appended) and its five Reuse layers take its index list with their own
    queries and windows.  per_layer[i] holds the inputs of CSA2 layer i (the
    encoder's layer i + 3): q_idx and w (Full layers only), q, win, out and
    an optional lse.  The two pure sliding-window layers in front (1 and 2)
    are not part of this path.  One workspace serves every layer in turn."""

    def __init__(self, csa, caches, qs, per_layer, *, k, n_win, max_n, sm_scale=1.0,
                 counters=None):
        import torch
        self.plan = encoder_csa2_layers()
        dev = per_layer[0]["q"].device
        nq = qs.nq
        n_blocks = 1 + max(p.cache for p in self.plan)
        assert len(caches) == n_blocks and len(per_layer) == len(self.plan)
        self.idx = [torch.zeros(nq, k, dtype=torch.int32, device=dev) for _ in range(n_blocks)]
        self.cnt = [torch.zeros(nq, dtype=torch.int32, device=dev) for _ in range(n_blocks)]
        ws = None
        self.layers = []
        for p, L in zip(self.plan, per_layer):
            full = p.mode == FULL
            layer = csa.Layer(csa.FULL if full else csa.REUSE, caches[p.cache], qs, k=k,
                              q=L["q"], win=L["win"], n_win=n_win, out=L["out"],
                              idx=self.idx[p.cache], cnt=self.cnt[p.cache],
                              q_idx=L.get("q_idx") if full else None,
                              w=L.get("w") if full else None, max_n=max_n, lse=L.get("lse"),
                              sm_scale=sm_scale, counters=counters, ws=ws)
            ws = layer.ws
            self.layers.append(layer)

    def __call__(self):
        for layer in self.layers:
            layer()
