"""Seeded synthetic inputs shaped like the pages' workloads.

This module is the one thing the CUDA path's tests/bench and the CPU oracle
share.  It holds none of the method's arithmetic: it draws numbers, rounds
them to the BF16 input format, and builds routing lists.  Every draw comes from
numpy's PCG64 seeded by SeedSequence([seed, config, tensor_id]).

Workload shapes (dense 8B-70B-class projections and a 30B-class MoE layer)
follow the serving workloads the pages describe; no dataset, evaluation suite
or trained weight is used or stood in for beyond these shapes and value
distributions:
  - activations ~ N(0, 1) with a fraction of K-columns ("outlier channels")
    multiplied by a factor (the pages describe activation outliers up to
    100x the mean);
  - weights ~ N(0, 0.02).
"""
import numpy as np

SEED = 0

# name -> shape/distribution recipe
CONFIGS = {
    1: dict(name="single_layer", M=128, N=256, K=512, outlier_frac=0.01, outlier_factor=50.0),
    2: dict(name="decode_mlp_up", Ms=(1, 8, 16), N=28672, K=8192, outlier_frac=0.005,
            outlier_factor=100.0),
    3: dict(name="prefill_proj", M=4096, Ns=(8192, 28672), K=8192, outlier_frac=0.005,
            outlier_factor=100.0),
    4: dict(name="policy_stack", layers=8, M=2048, N=4096, K=4096, outlier_frac=0.01,
            outlier_factor=50.0, n_sensitive=2),
    5: dict(name="moe_grouped", T=2048, H=2048, E=128, topk=8, inter=768, zipf_s=1.1,
            beta=0.17, outlier_frac=0.01, outlier_factor=50.0),
}


def rng(cfg: int, tensor_id: int, seed: int = SEED) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, cfg, tensor_id]))


def bf16_bits(f32: np.ndarray) -> np.ndarray:
    """Round finite float32 values to the nearest BF16 (ties to even) and
    return the 16-bit patterns."""
    u = np.ascontiguousarray(f32, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations(cfg: int, tensor_id: int, M: int, K: int, outlier_frac: float,
                outlier_factor: float, seed: int = SEED) -> np.ndarray:
    """BF16 bits [M, K]: N(0,1) with round(outlier_frac*K) distinct columns
    (drawn without replacement) multiplied by outlier_factor."""
    g = rng(cfg, tensor_id, seed)
    x = g.standard_normal((M, K), dtype=np.float32)
    n_out = int(round(outlier_frac * K))
    if n_out:
        cols = g.choice(K, n_out, replace=False)
        x[:, cols] *= np.float32(outlier_factor)
    return bf16_bits(x)


def weights(cfg: int, tensor_id: int, N: int, K: int, std: float = 0.02,
            seed: int = SEED) -> np.ndarray:
    """BF16 bits [N, K] drawn from N(0, std^2)."""
    g = rng(cfg, tensor_id, seed)
    w = g.standard_normal((N, K), dtype=np.float32) * np.float32(std)
    return bf16_bits(w)


def sensitive_flags(layers: int = 8, n_sensitive: int = 2, seed: int = SEED) -> np.ndarray:
    """0/1 per layer, n_sensitive of them set (seeded choice without replacement)."""
    g = rng(4, 99, seed)
    f = np.zeros(layers, np.uint8)
    f[g.choice(layers, n_sensitive, replace=False)] = 1
    return f


def moe_routing(T: int = 2048, E: int = 128, topk: int = 8, zipf_s: float = 1.1,
                beta: float = 0.17, literal: bool = False, seed: int = SEED):
    """Top-k expert routing from FP32 router logits with a Zipf(s) expert
    popularity.

    Default reading: logits[t, e] = beta * log p(rank(e)) + N(0, 1), with
    p(r) proportional to r^-s and ranks a seeded permutation of the experts;
    beta = 0.17 yields per-expert counts of roughly 70..400 for 2048 tokens.
    literal=True draws Plackett-Luce samples of the Zipf law itself
    (logits = log p + Gumbel), whose counts reach ~1850 (a stress case).

    Returns (row_idx int32 [T*topk], offsets int64 [E+1], counts int64 [E],
    logits float32 [T, E]): assignment j of expert e (offsets[e] <= j <
    offsets[e+1]) reads token row_idx[j]; tokens appear in increasing order
    within an expert."""
    g = rng(5, 100, seed)
    perm = g.permutation(E)
    ranks = np.arange(1, E + 1, dtype=np.float64)
    p = ranks ** (-zipf_s)
    p /= p.sum()
    logp = np.log(p[perm])
    if literal:
        logits = (logp[None, :] + g.gumbel(size=(T, E))).astype(np.float32)
    else:
        logits = (beta * logp[None, :] + g.standard_normal((T, E))).astype(np.float32)
    top = np.argsort(-logits, axis=1, kind="stable")[:, :topk]
    tok = np.repeat(np.arange(T, dtype=np.int64), topk)
    exp = top.reshape(-1).astype(np.int64)
    order = np.lexsort((tok, exp))
    row_idx = tok[order].astype(np.int32)
    counts = np.bincount(exp, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    return row_idx, offsets, counts, logits


def moe_gate_weights(logits, row_idx, offsets, topk: int = 8) -> np.ndarray:
    """Routing weight of every routed row (float32 [R]): the softmax of the
    token's top-k router logits, renormalised over the k chosen experts, for
    the (token row_idx[j], expert owning row j) pair."""
    logits = np.asarray(logits, np.float64)
    T, E = logits.shape
    top = np.argsort(-logits, axis=1, kind="stable")[:, :topk]
    sel = np.take_along_axis(logits, top, 1)
    w = np.exp(sel - sel.max(axis=1, keepdims=True))
    w /= w.sum(axis=1, keepdims=True)
    table = np.zeros((T, E))
    table[np.arange(T)[:, None], top] = w
    expert = np.repeat(np.arange(E), np.diff(np.asarray(offsets, np.int64)))
    return table[np.asarray(row_idx, np.int64), expert].astype(np.float32)


def moe_routing_from_counts(counts, T: int, seed: int = SEED):
    """Routing lists for prescribed per-expert counts (e.g. forced-empty
    experts): expert e takes counts[e] distinct tokens drawn without
    replacement, listed in increasing token order."""
    g = rng(5, 101, seed)
    counts = np.asarray(counts, np.int64)
    rows = [np.sort(g.choice(T, int(c), replace=False)) for c in counts]
    row_idx = (np.concatenate(rows) if rows else np.zeros(0)).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    return row_idx, offsets
