"""Seeded synthetic input streams (no GPU)."""
import numpy as np

from step_gpt_train_gb300 import data


def test_stream_is_deterministic_and_counter_based():
    a = data.token_stream("zipf", 5000, 1234)
    b = data.token_stream("zipf", 5000, 1234)
    assert np.array_equal(a, b)
    assert np.array_equal(data.token_stream("zipf", 100, 1234), a[:100])
    assert not np.array_equal(data.token_stream("zipf", 5000, 1235), a)


def test_uniform_stream_range():
    s = data.token_stream("uniform", 200_000, 3, vocab=512)
    assert s.min() == 0 and s.max() == 511
    counts = np.bincount(s, minlength=512)
    assert counts.std() / counts.mean() < 1.3 / np.sqrt(counts.mean())  # Poisson spread


def test_zipf_frequencies_match_pmf():
    n = 400_000
    s = data.token_stream("zipf", n, 11)
    assert s.min() >= 0 and s.max() < data.GPT2_VOCAB
    w = np.arange(1, data.GPT2_VOCAB + 1, dtype=np.float64) ** -1.1
    p = w / w.sum()
    counts = np.bincount(s, minlength=data.GPT2_VOCAB)
    for r in range(5):  # the heaviest ranks, e.g. id 0 at about 13.9 %
        sigma = np.sqrt(n * p[r] * (1 - p[r]))
        assert abs(counts[r] - n * p[r]) < 5 * sigma
    assert abs(p[0] - 0.139) < 0.001


def test_batches_shift_by_one():
    tok, tgt = data.batches("zipf", 3, 16, 4, 7)
    flat_t = tok.reshape(4, -1)
    flat_g = tgt.reshape(4, -1)
    assert np.array_equal(flat_t[:, 1:], flat_g[:, :-1])
    assert np.array_equal(flat_g[:-1, -1], flat_t[1:, 0])  # windows are contiguous
    s = data.token_stream("zipf", 4 * 48 + 1, 7)
    assert np.array_equal(tok.reshape(-1), s[:-1])


def test_eos_insertion():
    n = 300_000
    s = data.token_stream("zipf", n, 5, eos_every=700.0)
    pos = np.flatnonzero(s == data.GPT2_EOS)
    gaps = np.diff(pos) - 1
    assert abs(gaps.mean() - 700) < 30
    plain = data.token_stream("zipf", n, 5)
    base_rate = np.mean(plain == data.GPT2_EOS)
    assert len(pos) > n / 701 * 0.8 + base_rate * n


def test_round_to_bf16():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38], dtype=np.float32)
    r = data.round_to_bf16(x)
    assert r[0] == 1.0 and r[1] == 1.0  # tie to even
    assert r[2] == 1.0 + 4 * 2 ** -8  # tie to even (odd lsb rounds up)
    assert r[3] == -2.5
    assert np.all((r.view(np.uint32) & 0xFFFF) == 0)
