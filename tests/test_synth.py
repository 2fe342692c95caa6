"""Checks of the seeded input generator (input preparation, not the path)."""
import numpy as np

from qlora_fine_tuning_gb300 import synth


def test_codebooks_sorted_and_span_unit_interval():
    for kind in ("Q", "U"):
        cb = synth.codebook(kind)
        assert cb.dtype == np.float32 and cb.shape == (16,)
        assert np.all(np.diff(cb) > 0)
        assert cb[0] == -1.0 and cb[-1] == 1.0
    q = synth.codebook("Q").astype(np.float64)
    assert np.allclose(q, -q[::-1], atol=0)  # symmetric quantiles


def test_quantizer_picks_nearest_code_by_brute_force():
    rng = np.random.default_rng(0)
    cb = synth.codebook("Q")
    w = (rng.standard_normal((8, 128)) * 0.02).astype(np.float32)
    w[3, 64:] = 0.0  # a zero block
    idx, am = synth.quantize_4bit(w, cb)
    codes = np.empty((8, 128), dtype=np.int64)
    codes[:, 0::2] = idx & 0xF
    codes[:, 1::2] = idx >> 4
    blocks = w.reshape(-1, 64)
    assert np.array_equal(am, np.max(np.abs(blocks), axis=1))
    for b in range(blocks.shape[0]):
        a = float(am[b])
        for e in range(64):
            n, k = divmod(b * 64 + e, 128)
            t = 0.0 if a == 0 else float(w[n, k]) / a
            d = np.abs(t - cb.astype(np.float64))
            best = int(np.flatnonzero(d == d.min())[0])
            assert codes[n, k] == best


def test_generator_is_deterministic_and_shaped():
    a = synth.make_linear(64, 48, 128, 8, 2.0, seg_n=(16, 16, 16))
    b = synth.make_linear(64, 48, 128, 8, 2.0, seg_n=(16, 16, 16))
    for f in ("idx", "absmax", "X", "A", "B", "dY"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    assert a.idx.shape == (48, 64) and a.absmax.shape == (48 * 2,)
    assert a.X.shape == (64, 128) and a.A.shape == (128, 24) and a.B.shape == (8, 48)
    c = synth.make_linear(64, 48, 128, 8, 2.0, seg_n=(16, 16, 16), stream=1)
    assert not np.array_equal(a.X, c.X)


def test_packed_lengths_cover_the_batch():
    rng = np.random.default_rng(0)
    L = synth.packed_lengths(16384, rng)
    assert L.sum() == 16384 and L.min() >= 1 and L.max() <= 2048
    assert np.all(L[:-1] >= 64)


def test_flop_count_matches_the_definition():
    # 2MNK forward base + 2MNK dX base; three rank-r products on each side
    assert synth.flops_fwd_bwd(8192, 14336, 4096, 64) == 4 * 8192 * 14336 * 4096 + \
        6 * 8192 * 64 * (4096 + 14336)


def test_token_shards_share_the_layer_and_differ_in_tokens():
    a = synth.make_linear(16, 64, 64, 8, 1.0, seed=3)
    b = synth.make_linear(16, 64, 64, 8, 1.0, seed=3, shard=1)
    for k in ("idx", "absmax", "A", "B"):
        assert np.array_equal(getattr(a, k), getattr(b, k)), k
    assert not np.array_equal(a.X, b.X) and not np.array_equal(a.dY, b.dY)
