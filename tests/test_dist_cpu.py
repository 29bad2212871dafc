"""The multi-rank path on CPU (gloo, world size 2).

One fill is sharded by upper layer ([RF] "Ridge map": every upper layer has its
own map, norm and projections, and a filled entry depends only on x_S and that
layer's weights): rank r fills a contiguous block of the upper layers with no
data-path collective. These tests check that the blocks cover every (layer, row)
of the fill exactly once, that the ranks' oracle fills of their blocks, put
together, equal the oracle's fill of the whole problem bit for bit, that bench.py
under two gloo ranks plans exactly those blocks, and that the whole-job number is
every rank's units over the slowest rank's time."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle as O
import synth
from ridge_map_kv_gb300 import shard as sh

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

TINY = synth.FillConfig("tiny sharded fill", 97, d=32, L=7, S=2, N=24, T=5, H=2, hd=8, rope_theta=5e5,
                        exact="uniform10", lam=0.03, calib_n=0)        # P = 5: blocks of 3 and 2 on two ranks


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _f64_inputs(cfg):
    inp = synth.fill_inputs(cfg)
    f64 = O.bf16_bits_to_f64
    return {"x_S": f64(synth.bits(inp["x_S"])), "mask": synth.f32(inp["mask"]), "A": f64(synth.bits(inp["A"])),
            "b": synth.f32(inp["b"]).astype(np.float64), "gain": f64(synth.bits(inp["gain"])),
            "Wk": f64(synth.bits(inp["Wk"])), "Wv": f64(synth.bits(inp["Wv"]))}


def _oracle_fill(fields, t, L):
    zeros = np.zeros((L, fields["N"], fields["n_kv_heads"], fields["head_dim"]))
    kc, vc, idx = O.fill_kv(zeros, zeros, t["x_S"], t["mask"], t["A"], t["b"], t["gain"], t["Wk"], t["Wv"],
                            L=L, S=fields["S"], N=fields["N"], T=fields["T"], n_kv_heads=fields["n_kv_heads"],
                            head_dim=fields["head_dim"], rope_theta=fields["rope_theta"], rms_eps=fields["rms_eps"],
                            pos_offset=fields["pos_offset"])
    return kc, vc


@pytest.mark.parametrize("P", [0, 1, 5, 20, 48])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_layer_blocks_cover_every_upper_layer_once(P, world):
    blocks = [sh.layer_shard(P, 16, world, r) for r in range(world)]
    owner = np.full(P, -1)
    for b in blocks:
        assert 0 <= b.p0 <= b.p1 <= P
        assert np.all(owner[b.p0:b.p1] == -1), "a layer is in two blocks"
        owner[b.p0:b.p1] = b.rank
        assert list(b.model_layers) == list(range(16 + b.p0, 16 + b.p1))
    assert np.all(owner >= 0), "a layer is in no block"
    sizes = [b.layers for b in blocks]
    assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)
    assert all(blocks[r].p1 == blocks[r + 1].p0 for r in range(world - 1))   # contiguous, in rank order


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    ws, r = bench.dist_init("gloo")
    assert (ws, r) == (world, rank)
    # the rank's block as bench.py plans it, and the oracle's fill of that block alone
    block, fields = bench.fill_plan(TINY, ws, r, flags=4)
    t = sh.shard_weights(_f64_inputs(TINY), block)
    kc, vc = _oracle_fill(fields, t, fields["L"])
    bench.barrier()
    # rank 0 processed 1000 units per step in 50 ms, rank 1 the same in 80 ms
    timing = bench.aggregate_timing(1000, 10, 50.0 if rank == 0 else 80.0)
    out[rank] = {"block": (block.p0, block.p1, block.S), "fields": fields, "k": kc, "v": vc, "timing": timing}
    dist.destroy_process_group()


def test_two_gloo_ranks_fill_their_blocks_and_together_equal_the_whole_fill():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    cfg = TINY
    whole = dict(d=cfg.d, d_in=cfg.d_in, L=cfg.L, S=cfg.S, N=cfg.N, T=cfg.T, n_kv_heads=cfg.H, head_dim=cfg.hd,
                 rope_theta=cfg.rope_theta, rms_eps=cfg.rms_eps, pos_offset=cfg.pos_offset, flags=4)
    K, V = _oracle_fill(whole, _f64_inputs(cfg), cfg.L)
    Kg, Vg = np.zeros_like(K), np.zeros_like(V)
    for rank in (0, 1):
        o = out[rank]
        b = sh.layer_shard(cfg.P, cfg.S, 2, rank)
        assert o["block"] == (b.p0, b.p1, b.S)                       # bench plans the same blocks
        assert o["fields"] == sh.shard_desc_fields(whole, b)          # and the same descriptors
        assert o["fields"]["L"] == b.layers and o["fields"]["S"] == 0
        Kg[cfg.S + b.p0:cfg.S + b.p1] = o["k"]
        Vg[cfg.S + b.p0:cfg.S + b.p1] = o["v"]
        value, ms_per_step, t_max = o["timing"]
        assert t_max == 80.0
        assert ms_per_step == pytest.approx(8.0)
        assert value == pytest.approx(2 * 1000 * 10 / 0.080)
    assert [out[r]["block"][1] - out[r]["block"][0] for r in (0, 1)] == [3, 2]
    np.testing.assert_array_equal(Kg, K)
    np.testing.assert_array_equal(Vg, V)


def test_single_process_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    value, ms, t = bench.aggregate_timing(500, 4, 20.0)
    assert (value, ms, t) == (pytest.approx(100000.0), 5.0, 20.0)
    block, fields = bench.fill_plan(synth.DENSE27B, 1, 0, 0)
    assert (block.p0, block.p1) == (0, synth.DENSE27B.P) and fields["L"] == 48 and fields["S"] == 0
