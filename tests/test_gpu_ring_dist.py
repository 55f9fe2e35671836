"""The sequence-sharded ring (ring_dist) with the library's kernels: two ranks
as two processes on the one GPU, K/V and the travelling dK/dV exchanged over
gloo through host copies (no kernel of one rank waits on the other's). The
gathered result is held to the ring-vs-single-call bounds (fp32 outputs: the
forward out within the bf16 P-rounding bound, lse and gradients <= 1e-3)
against one call over the whole sequence, and sampled rows to the bf16-path
bound against the oracle."""

import os
import queue
import socket

import numpy as np
import pytest

import oracle
from blockwise_exact_attention_gb300 import workloads

from helpers import (TOL_LSE, TOL_RING, assert_close, assert_close_bf16, assert_within, report, ring_out_bound,
                     to_dev, to_np)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

L, H, HKV, D = 2048, 4, 2, 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, causal, window, results):
    import torch
    import torch.distributed as dist
    from blockwise_exact_attention_gb300 import ops, ring_dist
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        x = workloads.small_case(n=1, l=L, h=H, h_kv=HKV, d=D, is_causal=causal, window=window, seed=70)
        c = L // world
        sl = slice(rank * c, (rank + 1) * c)
        t = {k: torch.from_numpy(np.ascontiguousarray(x[k][:, sl])).cuda().to(torch.bfloat16)
             for k in ("q", "k", "v", "dout")}
        scale = 1.0 / np.sqrt(D)
        out, lse = ring_dist.ring_attention_fwd_sharded(t["q"], t["k"], t["v"], None, scale, causal, window)
        dq, dk, dv = ring_dist.ring_attention_bwd_sharded(t["dout"], t["q"], t["k"], t["v"], out, lse, None, scale,
                                                          causal, window)
        torch.cuda.synchronize()
        status = ops.device_status()
        results.put((rank, status, out.cpu().numpy(), lse.cpu().numpy(), dq.cpu().numpy(), dk.cpu().numpy(),
                     dv.cpu().numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("causal,window", [(True, (-1, -1)), (False, (-1, -1)), (True, (700, 0))])
def test_sharded_ring_on_one_gpu(causal, window):
    import blockwise_exact_attention_gb300 as bea
    import torch.multiprocessing as mp
    world = 2
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    pc = mp.start_processes(_worker, args=(world, _free_port(), causal, window, results), nprocs=world, join=False,
                            start_method="spawn")
    got = {}
    try:
        for _ in range(world):
            r = results.get(timeout=600)
            got[r[0]] = r[1:]
    except queue.Empty:
        pc.join(timeout=5)
        raise
    while not pc.join(timeout=60):
        pass
    assert all(got[r][0] == 0 for r in range(world))
    out = np.concatenate([got[r][1] for r in range(world)], axis=1)
    lse = np.concatenate([got[r][2] for r in range(world)], axis=2)
    dq, dk, dv = (np.concatenate([got[r][i] for r in range(world)], axis=1) for i in (3, 4, 5))
    # one call over the whole sequence, fp32 outputs
    x = workloads.small_case(n=1, l=L, h=H, h_kv=HKV, d=D, is_causal=causal, window=window, seed=70)
    q, k, v, do = (to_dev(x[s], torch.bfloat16) for s in ("q", "k", "v", "dout"))
    scale = 1.0 / np.sqrt(D)
    so, sl = bea.flash_mha_fwd(q, k, v, scale, causal, window, out_dtype=torch.float32)
    a_abs, _ = oracle.attention_fwd(x["q"], x["k"], np.abs(x["v"]), scale, causal, window)
    diff, _ = assert_within(out, to_np(so), ring_out_bound(a_abs), "sharded ring vs single out (fp32)")
    assert_close(lse, to_np(sl), TOL_RING, "sharded ring vs single lse")
    # the single-call backward from the same (out, lse) the ranks differentiated with
    ro_t = torch.from_numpy(np.ascontiguousarray(out)).float().cuda()
    rl_t = torch.from_numpy(np.ascontiguousarray(lse)).float().cuda()
    sg = bea.flash_mha_bwd(do, q, k, v, ro_t, rl_t, scale, causal, window, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), sg):
        assert_close(a, to_np(b), TOL_RING, name + " sharded ring vs single")
    rows = np.array([0, 1, 700, 1023, 1024, 1500, 2047])
    oo, ol = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal, window, rows=rows)
    assert_close_bf16(out[:, rows], oo, "sharded ring out vs oracle", output_is_bf16=False)
    assert_close(lse[:, :, rows], ol, TOL_LSE, "sharded ring lse vs oracle")
    report(f"[sharded ring, 2 ranks, causal={causal}, window={window}] max |ring - single| out {diff:.2e}")
