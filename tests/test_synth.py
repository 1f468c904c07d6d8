"""The shared seeded generator: determinism, distribution, bf16 rounding (CPU only)."""
import numpy as np
import torch

import synth
from synth import F32, BF16, KHIST, VHIST, Q
from synth import workloads


def test_counter_based_rows_are_position_independent():
    a = synth.rows(5, KHIST, 0, 3, 2, 0, 40, 16, F32)
    b = synth.rows(5, KHIST, 0, 3, 2, 17, 10, 16, F32)
    assert np.array_equal(a[17:27], b)
    assert not np.array_equal(a, synth.rows(5, VHIST, 0, 3, 2, 0, 40, 16, F32))
    assert not np.array_equal(a, synth.rows(6, KHIST, 0, 3, 2, 0, 40, 16, F32))


def test_history_pages_place_rows_by_logical_position():
    P, H, D, t = 16, 3, 8, 37
    pages = synth.history_pages(9, KHIST, 0, 1, 3, H, P, D, t, BF16)
    for h in range(H):
        r = synth.rows(9, KHIST, 0, 1, h, 0, t, D, BF16)
        for j in range(48):
            if j < t:
                assert np.array_equal(pages[j // P, h, j % P], r[j])
            else:
                assert not pages[j // P, h, j % P].any()


def test_values_are_standardised():
    x = synth.rows(1, Q, 0, 0, 0, 0, 200_000, 1, F32).ravel().astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert np.abs(x).max() <= 4 * 65535 / (2 * np.sqrt(4 * (65536.0 ** 2 - 1) / 12)) + 1e-6


def test_bf16_round_to_nearest_even_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(10000).astype(np.float32),
        np.array([0.0, -0.0, 1.0, np.inf, -np.inf, 1e-40, -3e-39, 3.4e38], np.float32),
        # exact ties: low half 0x8000 with even and odd kept bit
        np.array([0x3f808000, 0x3f818000, 0xbf808000, 0x00008000], np.uint32).view(np.float32),
    ])
    ours = synth.f32_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(synth.bf16_to_f32(ours),
                          torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_workload_recipes():
    w = workloads.batched()
    assert w.B == 64 and w.H == 32 and w.D == 128 and w.pool_pages == 32768
    assert w.seq_lens.min() >= 1 and w.seq_lens.max() <= 4096
    r = workloads.ragged()
    assert r.B == 256 and r.pool_pages == 600_000 and r.seq_lens.max() <= 32768
    assert 300 < np.median(r.seq_lens) < 900
    ops = workloads.churn_ops(r)
    assert len(ops) == 10_000 and ops == workloads.churn_ops(r)
    lc = workloads.long_context()
    assert (lc.seq_lens == 131072).all() and lc.pool_pages == 16 * 8192
    assert lc.kv_bytes() == 16 * 131072 * 8 * 128 * 2 * 2
