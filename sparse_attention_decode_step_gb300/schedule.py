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
