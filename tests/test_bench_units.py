"""The algorithmic units behind bench.py's rates, recomputed here from their
definitions: the FLOPs the sparse pattern requires (4 D per attended query-key
pair, valid keys only) and the bytes each HBM-bound step must move, on the
10 s FastH3 shape and, for the ragged-tile rule, by brute force on a tiny case.
The roofline fractions bench.py reports divide by these."""
import itertools

import numpy as np

import bench
from block_sparse_video_gb300.synthetic import CONFIGS, Config

D = 128
# the 10 s shape: batch 1, 56 heads, text 1,024 + audio 1,024 + video 72,576 tokens
P, LV, H, T, K = 2048, 72576, 56, 1134, 227


def test_shape_constants():
    c = CONFIGS["10s"]
    assert (c.batch, c.heads, c.prefix, c.len_video, c.n_video_tiles) == (1, H, P, LV, T)


def test_fine_and_coarse_flops_10s():
    fl = bench.effective_flops(CONFIGS["10s"])
    video_pairs = LV * (P + 64 * K)          # every video query: the prefix and its k selected tiles
    prefix_pairs = P * (P + LV)              # every prefix query: every key
    assert fl["fine"] == 4 * D * H * (video_pairs + prefix_pairs) == 38_874_923_401_216
    assert fl["coarse"] == 4 * D * H * T * T  # pooled scores and the coarse product, all tile pairs
    assert fl["total"] == fl["fine"] + fl["coarse"]


def test_ragged_tile_counts_its_valid_keys_only():
    """Brute force over every (query, key) pair of a tiny case whose last video
    tile holds 10 tokens, for a given selection."""
    c = Config("tiny ragged", 1, 2, 3, 2, 64 * 2 + 10, (0.5,), 0)
    t = c.n_video_tiles
    k = max(1, min(t, int(np.floor(0.5 * t + 0.5))))
    rng = np.random.default_rng(0)
    sel = np.stack([np.sort(rng.choice(t, size=k, replace=False)) for _ in range(c.heads * t)])
    sel = sel.reshape(1, c.heads, t, k)
    pairs = 0
    tile_of = lambda i: (i - c.prefix) // 64
    for h, i in itertools.product(range(c.heads), range(c.seq)):
        for j in range(c.seq):
            if i < c.prefix or j < c.prefix:      # prefix queries see every key; every query sees the prefix
                pairs += 1
            elif tile_of(j) in sel[0, h, tile_of(i)]:
                pairs += 1
    fl = bench.effective_flops(c, 0.5, tile_index=sel)
    assert fl["fine"] == 4 * D * pairs


def test_pool_and_coarse_bytes_10s():
    # pool: Q, K, V video rows read once (bf16), three fp32 [T, 128] means written per head
    assert bench.pool_bytes() == 3 * LV * H * D * 2 + 3 * H * T * D * 4 == 3_218_890_752
    # coarse + top-k: pooled Q, K, V read, int32 selections and the fp32 coarse rows written
    assert bench.coarse_bytes() == 3 * H * T * D * 4 + H * T * K * 4 + H * T * D * 4


def test_kv_stream_bytes_10s():
    """Every item loads its key tiles two at a time (128-key blocks of K and V,
    bf16): a video item its 32 prefix tiles and 227 selected ones (130 blocks,
    the last half empty), a prefix item all 32 + 1,134 tiles (583 blocks)."""
    blocks = H * (T * ((32 + K + 1) // 2) + 32 * ((32 + T + 1) // 2))
    assert blocks == 9_300_256
    assert bench.kv_stream_bytes() == blocks * 2 * 128 * D * 2


def test_subblock_counts_and_router_flops_10s():
    for s, k in ((0.75, 288), (0.8, 232)):
        kk, fine, router = bench.subblock_flops(CONFIGS["10s"], s)
        assert kk == k
        assert fine == 4 * D * H * (LV * (P + 64 * k) + P * (P + LV))
        assert router == 2 * D * H * (4 * T) ** 2   # every pair of 16-token sub-blocks


def test_clock_rejection_rule():
    """A timed region with a hardware or thermal slowdown, or SM clocks stuck
    well below maximum with no reason, is rejected; the power cap alone is kept."""
    ok = {"sm_mhz": 2010.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []})
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected({"sm_mhz": 2000.0, "sm_max_mhz": 2070.0, "reasons": [r, "sw_power_cap"]})
    assert bench.clocks_rejected({"sm_mhz": 1200.0, "sm_max_mhz": 2070.0, "reasons": []})
    assert not bench.clocks_rejected({"sm_mhz": 1200.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]})
    assert not bench.clocks_rejected({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]})
