"""Seeded synthetic inputs: token streams and test tensors.

This module only draws input data. It holds none of the training step's
arithmetic, so both the CUDA library's tests and the CPU oracle's tests take
their inputs from here.

The pages trained on TinyStories and FineWeb. Neither dataset is available,
so these seeded streams stand in for them, with the pages' shapes: GPT-2 ids
(V = 50257), T = 1024 windows, and a "next token" target stream
(llm.c "State of the Union", sections "Peak memory" and "Fine print").

Random bits come from splitmix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014): output i of the stream with
seed s is mix(s + (i+1) * 0x9E3779B97F4A7C15), where mix is the
Stafford-variant-13 finaliser. Output i therefore depends only on (s, i).
"""
from __future__ import annotations

import math

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)

GPT2_VOCAB = 50257
GPT2_VOCAB_PADDED = 50304
GPT2_EOS = 50256


def splitmix64_mix(z: np.ndarray) -> np.ndarray:
    """The splitmix64 output finaliser on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
    return z ^ (z >> np.uint64(31))


def splitmix64_stream(seed: int, start: int, n: int) -> np.ndarray:
    """Outputs start .. start+n-1 of the splitmix64 stream seeded with `seed`."""
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * GOLDEN
    return splitmix64_mix(state)


def uniform01(bits: np.ndarray) -> np.ndarray:
    """53-bit uniforms in [0, 1) from uint64 draws."""
    return (bits >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def zipf_cdf(n_ids: int, s: float) -> np.ndarray:
    """Cumulative probabilities of Zipf(s) on ranks 1..n_ids (rank r is id r-1)."""
    w = np.arange(1, n_ids + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    return cdf


def _inverse_cdf(cdf: np.ndarray, u: np.ndarray) -> np.ndarray:
    idx = np.searchsorted(cdf, u, side="right")
    return np.minimum(idx, len(cdf) - 1)


def _poisson_cdf(mean: float, cap: int) -> np.ndarray:
    k = np.arange(cap, dtype=np.float64)
    logp = -mean + k * math.log(mean) - np.array([math.lgamma(x + 1.0) for x in k])
    cdf = np.cumsum(np.exp(logp))
    cdf /= cdf[-1]
    return cdf


def token_stream(kind: str, n: int, seed: int, vocab: int = GPT2_VOCAB,
                 zipf_s: float = 1.1, eos_every: float | None = None,
                 eos_id: int = GPT2_EOS) -> np.ndarray:
    """The first n ids of one seeded synthetic token stream (int32).

    kind "uniform": i.i.d. ids, draw mod vocab.
    kind "zipf": i.i.d. Zipf(zipf_s) over ranks 1..vocab, rank r is id r-1,
      drawn by inverse CDF (binary search in a float64 CDF).
    eos_every: if set, an EoS id is inserted after every g ids, where the
      gaps g are Poisson(eos_every) draws from an independent stream (seed+1).
    """
    if kind == "uniform":
        ids = (splitmix64_stream(seed, 0, n) % np.uint64(vocab)).astype(np.int64)
    elif kind == "zipf":
        ids = _inverse_cdf(zipf_cdf(vocab, zipf_s), uniform01(splitmix64_stream(seed, 0, n)))
    else:
        raise ValueError(f"unknown stream kind {kind!r}")
    if eos_every is not None:
        cdf = _poisson_cdf(eos_every, int(eos_every * 4 + 64))
        n_gaps = n // max(1, int(eos_every // 2)) + 8
        gaps = _inverse_cdf(cdf, uniform01(splitmix64_stream(seed + 1, 0, n_gaps)))
        gaps = np.maximum(gaps, 1)
        out = np.empty(n, dtype=np.int64)
        pos, src, g = 0, 0, 0
        while pos < n:
            take = min(int(gaps[g]), n - pos)
            out[pos:pos + take] = ids[src:src + take]
            pos += take
            src += take
            g += 1
            if pos < n:
                out[pos] = eos_id
                pos += 1
        ids = out
    return ids.astype(np.int32)


def batches(kind: str, B: int, T: int, steps: int, seed: int, vocab: int = GPT2_VOCAB,
            eos_every: float | None = None):
    """tokens, targets of shape [steps, B, T] (int32) from one contiguous stream.

    Step k reads the window of B*T + 1 ids starting at k*B*T:
    tokens[k, b, t] = s[k*B*T + b*T + t] and targets = the same window shifted by one.
    """
    n = steps * B * T + 1
    s = token_stream(kind, n, seed, vocab=vocab, eos_every=eos_every)
    tok = np.empty((steps, B, T), dtype=np.int32)
    tgt = np.empty((steps, B, T), dtype=np.int32)
    for k in range(steps):
        base = k * B * T
        tok[k] = s[base:base + B * T].reshape(B, T)
        tgt[k] = s[base + 1:base + B * T + 1].reshape(B, T)
    return tok, tgt


def normal(seed: int, shape, std: float = 1.0, dtype=np.float32) -> np.ndarray:
    """Seeded N(0, std^2) test tensor (numpy PCG64); for per-kernel test inputs."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(size=shape) * std).astype(dtype)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), returned as float32.

    Used to make test inputs exactly representable in bf16, so both sides see
    the same values.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    out = r.astype(np.uint32).view(np.float32)
    return np.where(np.isnan(x), x, out)


# Workload presets, with the shapes of the pages' GPT-2 runs (T = 1024, GPT-2 vocab).
WORKLOADS = {
    "tiny": dict(n_layer=2, n_embd=64, n_head=4, vocab=512, vocab_padded=512, max_T=64,
                 B=4, T=64, mode=0, stream="uniform", eos_every=None),
    "124m-b8": dict(n_layer=12, n_embd=768, n_head=12, vocab=GPT2_VOCAB,
                    vocab_padded=GPT2_VOCAB_PADDED, max_T=1024, B=8, T=1024, mode=1,
                    stream="zipf", eos_every=None),
    "124m-b32": dict(n_layer=12, n_embd=768, n_head=12, vocab=GPT2_VOCAB,
                     vocab_padded=GPT2_VOCAB_PADDED, max_T=1024, B=32, T=1024, mode=1,
                     stream="zipf", eos_every=700.0),
    "350m-b16": dict(n_layer=24, n_embd=1024, n_head=16, vocab=GPT2_VOCAB,
                     vocab_padded=GPT2_VOCAB_PADDED, max_T=1024, B=16, T=1024, mode=1,
                     stream="zipf", eos_every=None),
    "1p5b-b8": dict(n_layer=48, n_embd=1600, n_head=25, vocab=GPT2_VOCAB,
                    vocab_padded=GPT2_VOCAB_PADDED, max_T=1024, B=8, T=1024, mode=1,
                    stream="zipf", eos_every=None),
}


def workload_batches(name: str, steps: int, seed: int = 1234, B: int | None = None,
                     T: int | None = None):
    w = WORKLOADS[name]
    B = w["B"] if B is None else B
    T = w["T"] if T is None else T
    return batches(w["stream"], B, T, steps, seed, vocab=w["vocab"], eos_every=w["eos_every"])
