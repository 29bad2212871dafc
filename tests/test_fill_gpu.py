"""GPU parity of rf_fill_kv against the fp64 oracle (through the C ABI).

Small cases compare every filled entry and check the whole cache bit for bit
against NaN canaries. They span several M/N tiles, ragged tails and the
degenerate arms. Full-size cases use the workloads' own shapes: bookkeeping on
the whole cache, values on sampled rows (first, last, neighbours of exact blocks,
the last prefix row and seeded random rows).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import ridge_map_kv_gb300 as rf
import synth
from fillcheck import assert_bookkeeping, assert_values, run_fill

pytestmark = pytest.mark.gpu


def _small(name, **kw):
    base = dict(name=name, index=90, d=512, L=5, S=2, N=400, T=37, H=2, hd=128, rope_theta=5e5,
                exact="uniform10", lam=0.03, calib_n=0)
    base.update(kw)
    return synth.FillConfig(**base)


def _mask_np(inp):
    return None if inp["mask"] is None else inp["mask"].cpu().numpy()


KERNELS = pytest.mark.parametrize("flags", [rf.RF_FLAG_SINGLE_CTA, rf.RF_FLAG_CTA_PAIR], ids=["single-cta", "cta-pair"])


@KERNELS
def test_toy_fill_matches_oracle_everywhere(flags):
    cfg = synth.TOY
    inp = synth.fill_inputs(cfg)
    res = run_fill(cfg, inp, flags=flags)
    assert res["status"] == 0
    idx = O.prefix_partition(cfg.N, cfg.T, _mask_np(inp))
    assert idx.tolist() == [0, 1, 2, 3, 8]
    assert res["n_fill"] == 5
    assert_bookkeeping(cfg, res, _mask_np(inp))
    assert_values(cfg, inp, res, idx)


@pytest.mark.parametrize("cfg", [
    _small("ragged 3 M-tiles, 2 N-tiles, hd128"),
    _small("hd64, 4 heads, 2 layers", d=768, L=4, S=2, N=300, T=20, H=4, hd=64, exact="blocks16_5"),
    _small("one layer, no exact rows", d=256, L=3, S=2, N=129, T=0, H=1, hd=128, exact=None),
    _small("position offset", d=256, L=4, S=1, N=200, T=8, H=2, hd=64, exact="uniform10", pos_offset=1000),
    _small("positions near 2^26", d=256, L=3, S=1, N=300, T=8, H=2, hd=128, exact="uniform10",
           pos_offset=(1 << 26) + 777),
], ids=lambda c: c.name)
@KERNELS
def test_fill_small_shapes_match_oracle(cfg, flags):
    inp = synth.fill_inputs(cfg)
    res = run_fill(cfg, inp, flags=flags)
    assert res["status"] == 0
    idx = O.prefix_partition(cfg.N, cfg.T, _mask_np(inp))
    assert res["n_fill"] == len(idx)
    assert_bookkeeping(cfg, res, _mask_np(inp))
    assert_values(cfg, inp, res, idx)


@KERNELS
def test_prefolded_weights_give_the_same_caches_bit_for_bit(flags):
    """Projections folded once by rf_fold_kv_weights (RF_WEIGHTS_PREFOLDED) and the
    gain folded inside the call give the same caches, bit for bit."""
    cfg = _small("prefolded vs folded in the call")
    inp = synth.fill_inputs(cfg)
    a = run_fill(cfg, inp, flags=flags)
    b = run_fill(cfg, inp, flags=flags, prefolded=True)
    assert a["status"] == 0 and b["status"] == 0
    assert torch.equal(a["kc"].view(torch.int16), b["kc"].view(torch.int16))
    assert torch.equal(a["vc"].view(torch.int16), b["vc"].view(torch.int16))


@pytest.mark.parametrize("case", ["all_exact", "tail_is_everything", "no_upper_layers", "one_row", "two_tiles_plus_one"])
def test_fill_degenerate_arms(case):
    cfg = _small(case, d=256, L=4, S=2, N=140, T=10, H=2, hd=64, exact=None)
    mask = None
    if case == "all_exact":
        mask = torch.ones(cfg.N - cfg.T, dtype=torch.uint8)
    elif case == "tail_is_everything":
        cfg = dataclasses.replace(cfg, T=cfg.N)
    elif case == "no_upper_layers":
        cfg = dataclasses.replace(cfg, S=cfg.L)
    elif case == "one_row":
        mask = torch.ones(cfg.N - cfg.T, dtype=torch.uint8)
        mask[77] = 0
    elif case == "two_tiles_plus_one":
        cfg = dataclasses.replace(cfg, N=267, T=10)
    inp = synth.fill_inputs(cfg)
    inp["mask"] = mask
    res = run_fill(cfg, inp)
    assert res["status"] == 0
    mnp = None if mask is None else mask.numpy()
    idx = O.prefix_partition(cfg.N, cfg.T, mnp)
    assert res["n_fill"] == len(idx)
    assert_bookkeeping(cfg, res, mnp)
    if len(idx) and cfg.P > 0:
        assert_values(cfg, inp, res, idx)


@pytest.mark.parametrize("offset", [0, 1, 3, 4])
def test_compaction_over_several_mask_tiles_at_any_mask_alignment(offset):
    """The compaction reads the mask 4 bytes per thread in tiles of 4096 rows, with
    32-bit loads where the mask is 4-byte aligned and byte loads elsewhere. A prefix
    of 3 tiles less one row, its mask at byte offsets 0..4 into a buffer: fill_idx
    (the workspace's first region) must equal the oracle's partition exactly, and the
    cache bookkeeping must hold bit for bit."""
    cfg = _small("compaction tiles", d=256, L=2, S=1, N=12300, T=13, H=2, hd=64, exact=None)
    n_prefix = cfg.N - cfg.T                                    # 12,287 = 3 * 4096 - 1
    rng = np.random.default_rng(17)
    mnp = (rng.random(n_prefix) < 0.3).astype(np.uint8)
    mnp[4090:4110] = 1                                          # an exact run across a tile edge
    mnp[-5:] = 0
    buf = torch.zeros(n_prefix + 8, dtype=torch.uint8, device="cuda")
    buf[offset:offset + n_prefix] = torch.as_tensor(mnp, device="cuda")
    inp = synth.fill_inputs(cfg)
    res = run_fill(cfg, inp, mask=buf[offset:offset + n_prefix])
    assert res["status"] == 0
    idx = O.prefix_partition(cfg.N, cfg.T, mnp)
    assert res["n_fill"] == len(idx)
    got = res["ws"][: n_prefix * 4].view(torch.int32)[: len(idx)].cpu().numpy()
    assert np.array_equal(got, idx)
    assert_bookkeeping(cfg, res, mnp)


def _sample_rows(idx: np.ndarray, mask_np, n_prefix: int, n_random=192, seed=1):
    rng = np.random.default_rng(seed)
    pick = {int(idx[0]), int(idx[-1])}
    if n_prefix - 1 in set(idx.tolist()):
        pick.add(n_prefix - 1)
    if mask_np is not None:
        ex = np.nonzero(mask_np)[0]
        fill = set(idx.tolist())
        for t in np.concatenate([ex - 1, ex + 1]):
            if 0 <= t < n_prefix and int(t) in fill:
                pick.add(int(t))
    pick = sorted(pick)
    rest = rng.choice(idx, size=min(n_random, len(idx)), replace=False)
    rows = np.unique(np.concatenate([rng.permutation(np.array(pick))[:64], rest]))
    return rows.astype(np.int64)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["llama8b", "qwen3_8b", "dense27b"])
@KERNELS
def test_fill_full_size_sampled(name, flags):
    cfg = synth.FILL_CONFIGS[name]
    inp = synth.fill_inputs(cfg, device="cuda")
    res = run_fill(cfg, inp, flags=flags)
    assert res["status"] == 0
    mnp = _mask_np(inp)
    idx = O.prefix_partition(cfg.N, cfg.T, mnp)
    assert res["n_fill"] == len(idx)
    assert_bookkeeping(cfg, res, mnp)
    rows = _sample_rows(idx, mnp, cfg.N - cfg.T)
    assert_values(cfg, inp, res, rows)


# --------------------------------------------------------------------------- #
# Key normalisation (per-head RMSNorm of K before RoPE, "Qwen models normalize keys")
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("cfg", [
    _small("key norm, hd128, ragged 3 M-tiles"),
    _small("key norm, hd64, 4 heads", d=768, L=4, S=2, N=300, T=20, H=4, hd=64, exact="blocks16_5"),
], ids=lambda c: c.name)
@KERNELS
def test_fill_with_key_norm_matches_oracle(cfg, flags):
    inp = synth.fill_inputs(cfg)
    kg = synth.key_norm_gain(cfg)
    res = run_fill(cfg, inp, flags=flags, k_norm_gain=kg)
    assert res["status"] == 0
    mnp = _mask_np(inp)
    idx = O.prefix_partition(cfg.N, cfg.T, mnp)
    assert_bookkeeping(cfg, res, mnp)
    assert_values(cfg, inp, res, idx, k_norm_gain=kg)


@pytest.mark.slow
def test_fill_with_key_norm_qwen3_shape_sampled():
    """Qwen3-8B shape (d=4096, 23 upper layers, N=32768, no exact rows) with key
    normalisation: bookkeeping on the whole cache, values on sampled rows."""
    cfg = synth.FILL_CONFIGS["qwen3_8b"]
    inp = synth.fill_inputs(cfg, device="cuda")
    kg = synth.key_norm_gain(cfg, device="cuda")
    res = run_fill(cfg, inp, k_norm_gain=kg)
    assert res["status"] == 0
    mnp = _mask_np(inp)
    idx = O.prefix_partition(cfg.N, cfg.T, mnp)
    assert res["n_fill"] == len(idx)
    assert_bookkeeping(cfg, res, mnp)
    assert_values(cfg, inp, res, _sample_rows(idx, mnp, cfg.N - cfg.T), k_norm_gain=kg)


# --------------------------------------------------------------------------- #
# Non-square maps: x_S and the map input are d_in wide, x̂ and the projections d
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("cfg", [
    _small("d_in 1024 -> d 256 (4 streams)", d=256, d_in=1024, L=4, S=2, N=300, T=20, H=2, hd=64),
    _small("d_in 768 -> d 512, hd128, ragged", d=512, d_in=768),
], ids=lambda c: c.name)
@KERNELS
def test_fill_with_non_square_maps_matches_oracle(cfg, flags):
    inp = synth.fill_inputs(cfg)
    assert inp["x_S"].shape[1] == cfg.d_in and inp["A"].shape[1:] == (cfg.d, cfg.d_in)
    res = run_fill(cfg, inp, flags=flags)
    assert res["status"] == 0
    mnp = _mask_np(inp)
    idx = O.prefix_partition(cfg.N, cfg.T, mnp)
    assert res["n_fill"] == len(idx)
    assert_bookkeeping(cfg, res, mnp)
    assert_values(cfg, inp, res, idx)


@pytest.mark.slow
def test_fill_flash_next_shaped_maps_sampled():
    """Flash-Next-shaped maps: 24 upper layers of 10,240 -> 2,560, N = 32,768,
    T = 2,048 (KV heads 2 x 128: the pages do not give them)."""
    cfg = synth.FILL_CONFIGS["flash_next"]
    inp = synth.fill_inputs(cfg, device="cuda")
    res = run_fill(cfg, inp)
    assert res["status"] == 0
    mnp = _mask_np(inp)
    idx = O.prefix_partition(cfg.N, cfg.T, mnp)
    assert res["n_fill"] == len(idx)
    assert_bookkeeping(cfg, res, mnp)
    assert_values(cfg, inp, res, _sample_rows(idx, mnp, cfg.N - cfg.T))


# --------------------------------------------------------------------------- #
# Layer shards: the blocks of a multi-GPU fill, run one after another here
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("world", [2, 3])
def test_layer_blocks_filled_separately_equal_the_whole_fill(world):
    """Each rank of a sharded fill calls rf_fill_kv on its block of upper layers as a
    fill of its own (L = its layer count, S = 0, a cache of just those layers, its
    slices of the maps and projections). Run block by block on one GPU, the blocks'
    caches put together equal the whole fill's upper layers bit for bit."""
    from ridge_map_kv_gb300 import shard as sh
    cfg = _small("sharded by layer", L=7, S=2)
    inp = synth.fill_inputs(cfg)
    whole = run_fill(cfg, inp, canary=False)       # zero caches: entries never written stay 0 in both
    assert whole["status"] == 0
    for r in range(world):
        b = sh.layer_shard(cfg.P, cfg.S, world, r)
        part = dataclasses.replace(cfg, L=b.layers, S=0)
        res = run_fill(part, sh.shard_weights(inp, b), canary=False)
        assert res["status"] == 0 and res["n_fill"] == whole["n_fill"]
        for key in ("kc", "vc"):
            assert torch.equal(res[key].view(torch.int16), whole[key][cfg.S + b.p0:cfg.S + b.p1].view(torch.int16))
