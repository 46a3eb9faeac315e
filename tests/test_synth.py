"""The seeded input generator: reproducible, and planted blocks avoid the forced blocks."""
import numpy as np
import torch

import synth


def test_draws_are_seeded_and_bf16():
    a = synth.normal_bf16((4, 5), 3, 1)
    b = synth.normal_bf16((4, 5), 3, 1)
    c = synth.normal_bf16((4, 5), 3, 2)
    assert a.dtype == torch.bfloat16 and torch.equal(a, b) and not torch.equal(a, c)


def test_planted_blocks_avoid_block0_and_tail():
    for seed in range(20):
        blk = synth.planted_blocks(seed, 64, 8, 0, 1)
        assert len(set(blk.tolist())) == 8 and blk.min() >= 1 and blk.max() <= 62


def test_plant_shifts_only_planted_rows_along_direction():
    K = torch.zeros(64 * 6, 4, dtype=torch.bfloat16)
    synth.plant(K, [2, 4], np.array([0.0, 3.0, 0.0, 4.0]))
    rows = K.double()
    assert torch.all(rows[128:192] == torch.tensor([0.0, 0.3, 0.0, 0.4], dtype=torch.float64).to(torch.bfloat16).double())
    assert torch.all(rows[:128] == 0) and torch.all(rows[192:256] == 0)


def test_plant_batched_matches_plant():
    K1 = synth.normal_bf16((2, 2, 640, 8), 1, 1)
    K2 = K1.clone()
    blocks = np.array([[[1, 3], [2, 8]], [[5, 6], [1, 2]]])
    dirs = torch.randn(2, 2, 8, dtype=torch.float64)
    synth.plant_batched(K1, blocks, dirs)
    for b in range(2):
        for g in range(2):
            synth.plant(K2[b, g], blocks[b, g], dirs[b, g].numpy())
    assert torch.equal(K1, K2)
