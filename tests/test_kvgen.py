"""The seeded input generator: the numpy and torch implementations agree bit for bit, rows can be
regenerated individually, and the workloads have the stated structure."""
import numpy as np
import torch

import kvgen


def test_numpy_and_torch_agree():
    idx = np.arange(0, 1 << 18, dtype=np.int64) * 7919 % (1 << 31)
    a = kvgen.normal_fp16_np(5, kvgen.TAG_K, idx, sub=3)
    b = kvgen.normal_fp16_torch(5, kvgen.TAG_K, torch.from_numpy(idx), sub=3).numpy()
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    w = kvgen.words_np(1, 2, idx)
    wt = kvgen.words_torch(1, 2, torch.from_numpy(idx)).numpy()
    assert np.array_equal(w.astype(np.int64), wt)


def test_kv_spec_rows_full_and_torch_agree():
    spec = kvgen.KVSpec(seed=0, layer=3, is_key=True, n_seq=2, n_tok=40, num_heads=4,
                        head_dim=64)
    full = spec.full_np()
    t = spec.full_torch("cpu", chunk_rows=37).numpy()
    assert np.array_equal(full.view(np.uint16), t.view(np.uint16))
    rows = np.array([0, 5, 77, 319])
    assert np.array_equal(spec.rows_np(rows).view(np.uint16),
                          full.reshape(-1, 64)[rows].view(np.uint16))
    # zero rows: token 0, head 0 of every sequence (keys)
    assert np.all(full[0, 0] == 0) and np.all(full[40, 0] == 0)
    # outlier channels are ~10x larger
    ch = kvgen.outlier_channels(0, 3, 4, 64, 4)
    mags = np.abs(full.astype(np.float32)).mean(axis=0)
    for h in range(4):
        other = np.setdiff1d(np.arange(64), ch[h])
        assert mags[h, ch[h]].min() > 5 * mags[h, other].max()


def test_values_zero_row_is_last_token_last_head():
    spec = kvgen.KVSpec(seed=1, layer=0, is_key=False, n_seq=3, n_tok=10, num_heads=4,
                        head_dim=16)
    full = spec.full_np()
    for s in range(3):
        assert np.all(full[s * 10 + 9, 3] == 0)
    assert np.count_nonzero(np.all(full == 0, axis=-1)) == 3


def test_kivi_spec_agrees_and_has_outliers():
    spec = kvgen.KiviSpec(seed=3, layer=1, is_key=True, batch=2, num_heads=2, seq=64, head_dim=64)
    full = spec.full_np()
    t = spec.full_torch("cpu", chunk_rows=50).numpy()
    assert np.array_equal(full.view(np.uint16), t.view(np.uint16))
    assert np.array_equal(spec.slab_np(1, 1, 10, 20).view(np.uint16),
                          full[1, 1, 10:20].view(np.uint16))


def test_quantile_table_against_an_independent_inverse_cdf():
    """The table's nodes are standard normal quantiles: compared with the standard library's
    NormalDist (a different algorithm) at nodes across the whole range, tails included."""
    from statistics import NormalDist
    t, slope = kvgen.quantile_table()
    nd = NormalDist()
    n = t.size
    for k in list(range(0, 64)) + list(range(n - 64, n)) + list(range(0, n, 4099)):
        want = nd.inv_cdf((k * 4096 + 0.5) / 2.0 ** 32)
        assert abs(float(t[k]) - want) <= 2e-7 * max(1.0, abs(want)), k
    assert np.all(slope > 0)                              # monotone
    top = float(t[-1]) + 4095.0 * float(slope[-1])        # the node at the largest word, 2^32 - 1
    assert abs(float(t[0]) + top) < 1e-5                  # symmetric ends


def test_moments_and_permutation():
    x = kvgen.normal_fp16_np(0, 1, np.arange(1 << 22)).astype(np.float64)
    assert abs(x.mean()) < 2e-3 and abs(x.std() - 1) < 2e-3
    kurt = np.mean((x - x.mean()) ** 4) / x.var() ** 2
    assert abs(kurt - 3.0) < 0.02                         # Gaussian, not bounded Irwin-Hall (2.7)
    # Gaussian tails: P(|z| > 4) = 6.3e-5 (about 265 of 4 Mi draws)
    tail = int(np.count_nonzero(np.abs(x) > 4.0))
    assert 180 < tail < 360
    assert np.abs(x).max() > 4.5
    pt = kvgen.random_page_table(1, 8, 100)
    assert sorted(pt.ravel().tolist()) == list(range(800))
    lens = kvgen.decode_append_lengths(2, 64)
    assert lens.min() >= 1024 and lens.max() <= 65536
    q = kvgen.queries_np(0, 2, 1, 24, 256)
    qt = kvgen.queries_torch(0, 2, 1, 24, 256, "cpu").numpy()
    assert np.array_equal(q.view(np.uint16), qt.view(np.uint16))
