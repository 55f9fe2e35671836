"""The sequence-sharded ring (ring_dist) on CPU ranks over gloo: its schedule,
K/V exchange, causal/window skipping and travelling dK/dV accumulators,
driven with an fp64 restatement of the per-step compute (the oracle's block
attention, merge and backward), against the oracle's single-call attention of
the whole sequence."""

import os
import socket

import numpy as np
import pytest
import torch

import oracle
from blockwise_exact_attention_gb300 import ring_dist, workloads


class OracleStep:
    """The per-step compute of ring_dist restated with the fp64 oracle (test only)."""

    def fwd_first(self, q, k, v, out, lse, scale, causal, window):
        o, l = oracle.attention_fwd(q.numpy(), k.numpy(), v.numpy(), scale, causal, window, key_offset=0)
        out.copy_(torch.from_numpy(o))
        lse.copy_(torch.from_numpy(l))

    def fwd_merge(self, q, k, v, out, lse, scale, causal, window, key_offset):
        o, l = oracle.attention_fwd(q.numpy(), k.numpy(), v.numpy(), scale, causal, window, key_offset=key_offset)
        mo, ml = oracle.merge_max_form(out.double().numpy(), lse.double().numpy(), o, l)
        out.copy_(torch.from_numpy(mo))
        lse.copy_(torch.from_numpy(ml))

    def bwd_begin(self, dout, out, lse):
        self.saved = (out.double().numpy(), lse.double().numpy())
        self.dq = np.zeros(dout.shape)

    def bwd_pair(self, dout, q, k, v, dk, dv, scale, causal, window, key_offset):
        out, lse = self.saved
        gq, gk, gv = oracle.attention_bwd(dout.numpy(), q.numpy(), k.numpy(), v.numpy(), out, lse, scale, causal,
                                          window, key_offset=key_offset)
        self.dq += gq
        dk += torch.from_numpy(gk).to(dk.dtype)
        dv += torch.from_numpy(gv).to(dv.dtype)

    def bwd_end(self, dq, scale):
        dq.copy_(torch.from_numpy(self.dq))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, causal, window, results):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        L, h, hkv, d = 24 * world, 2, 1, 16
        x = workloads.small_case(n=1, l=L, h=h, h_kv=hkv, d=d, is_causal=causal, window=window, seed=7 + world)
        c = L // world
        sl = slice(rank * c, (rank + 1) * c)
        scale = 1.0 / np.sqrt(d)
        t = {key: torch.from_numpy(np.ascontiguousarray(x[key][:, sl])).double() for key in ("q", "k", "v", "dout")}
        out, lse = ring_dist.ring_attention_fwd_sharded(t["q"], t["k"], t["v"], None, scale, causal, window,
                                                        step=OracleStep())
        # the backward from the final (out, lse) of the local queries
        dq, dk, dv = ring_dist.ring_attention_bwd_sharded(t["dout"], t["q"], t["k"], t["v"], out, lse, None, scale,
                                                          causal, window, step=OracleStep())
        results.put((rank, out.double().numpy(), lse.double().numpy(), dq.double().numpy(), dk.double().numpy(),
                     dv.double().numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,causal,window", [(2, True, (-1, -1)), (2, False, (-1, -1)), (3, True, (-1, -1)),
                                                 (3, True, (30, 0)), (2, False, (10, 7)), (4, False, (-1, 5))])
def test_sharded_ring_matches_single_call(world, causal, window):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    pc = mp.start_processes(_worker, args=(world, _free_port(), causal, window, results), nprocs=world, join=False,
                            start_method="spawn")
    got = dict()
    import queue
    try:
        for _ in range(world):   # read before joining: a child blocks on a full pipe until its result is taken
            r = results.get(timeout=180)
            got[r[0]] = r[1:]
    except queue.Empty:
        pc.join(timeout=5)   # raises the failing child's exception if there is one
        raise
    while not pc.join(timeout=60):
        pass
    L, h, hkv, d = 24 * world, 2, 1, 16
    x = workloads.small_case(n=1, l=L, h=h, h_kv=hkv, d=d, is_causal=causal, window=window, seed=7 + world)
    scale = 1.0 / np.sqrt(d)
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal, window)
    c = L // world
    out = np.concatenate([got[r][0] for r in range(world)], axis=1)
    lse = np.concatenate([got[r][1] for r in range(world)], axis=2)
    assert np.abs(out - ro).max() <= 1e-6
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(lse), fin) and np.abs(lse[fin] - rl[fin]).max() <= 1e-6
    # gradients: each rank's dq of its queries, dk/dv of its own key chunk (brought home)
    rdq, rdk, rdv = oracle.attention_bwd(x["dout"], x["q"], x["k"], x["v"], out, lse, scale, causal, window)
    for i, ref in ((2, rdq), (3, rdk), (4, rdv)):
        g = np.concatenate([got[r][i] for r in range(world)], axis=1)
        assert np.abs(g - ref).max() <= 1e-5, (i, np.abs(g - ref).max())
    assert c * world == L


def test_band_has_keys_matches_the_oracle_mask():
    rng = np.random.default_rng(3)
    for _ in range(200):
        c = int(rng.integers(1, 9))
        causal = bool(rng.integers(0, 2))
        window = (int(rng.integers(-1, 12)), int(rng.integers(-1, 12)))
        if causal and window[1] > 0:
            window = (window[0], 0)
        koff = int(rng.integers(-30, 30))
        want = oracle.visible_mask(np.arange(c), c, causal, window, koff).any()
        assert ring_dist.band_has_keys(c, causal, window, koff) == bool(want)
