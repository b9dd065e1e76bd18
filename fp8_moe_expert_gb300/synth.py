"""Seeded synthetic inputs for the MoE expert path.

This module draws random numbers and rounds them to bf16; it holds none of the
quantizers' or GEMMs' arithmetic.  Both the CUDA path (tests, bench) and the CPU
oracle take their inputs from here, and nothing else is shared between them.

Workloads follow the expert shapes of "Scaling and Optimizing Frontier Model
Training" ("MXFP8 expert kernels": 32 experts per rank, hidden 7168,
intermediate 2048).  Each generator's docstring states its recipe.

Two back ends:
  * numpy (``np.random.default_rng(seed)``, PCG64) for everything the CPU
    oracle must see in full: the tiny case, the quantizer batch, expert loads;
  * torch on the GPU (``torch.Generator(device).manual_seed(seed)``) for the
    multi-GB activation and weight tensors of the full-size MoE workloads;
    parity checks copy the rows they sample back to the host.
"""
from __future__ import annotations

import numpy as np

HIDDEN = 7168
INTERMEDIATE = 2048
EXPERTS = 32


# ---------------------------------------------------------------- bf16 bits --
def bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounding = 0x7FFF + ((u >> 16) & 1)
    out = ((u + rounding) >> 16).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_np(t) -> np.ndarray:
    """A torch bf16 tensor (any device) -> its uint16 bit patterns as numpy."""
    import torch

    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_float(bits) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# -------------------------------------------------------------- expert loads --
def offsets_from_counts(counts) -> np.ndarray:
    counts = np.asarray(counts, dtype=np.int64)
    off = np.zeros(len(counts) + 1, dtype=np.int64)
    np.cumsum(counts, out=off[1:])
    return off.astype(np.int32)


def dirichlet_counts(rows: int = 65536, experts: int = EXPERTS, seed: int = 2) -> np.ndarray:
    """Expert loads: p ~ Dirichlet(1, ..., 1), counts ~ Multinomial(rows, p)."""
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.ones(experts))
    return rng.multinomial(rows, p).astype(np.int64)


def zipf_counts(rows: int = 262144, experts: int = EXPERTS, s: float = 1.2, empty: int = 3,
                seed: int = 4) -> np.ndarray:
    """Skewed loads: Zipf(s) over a seeded order of the non-empty experts, ``empty``
    seeded experts forced to zero rows, and no count a multiple of 128."""
    rng = np.random.default_rng(seed)
    empty_ids = rng.choice(experts, size=empty, replace=False)
    live = np.array([e for e in range(experts) if e not in set(empty_ids.tolist())])
    order = rng.permutation(live)
    weights = np.arange(1, len(order) + 1, dtype=np.float64) ** (-s)
    p = np.zeros(experts)
    p[order] = weights / weights.sum()
    counts = rng.multinomial(rows, p).astype(np.int64)
    # move single rows so that no live count is a multiple of 128
    for _ in range(10 * experts):
        bad = [e for e in live if counts[e] % 128 == 0]
        if not bad:
            break
        e = bad[0]
        j = live[(list(live).index(e) + 1) % len(live)]
        if counts[e] > 0:
            counts[e] -= 1
            counts[j] += 1
        else:
            counts[j] -= 1
            counts[e] += 1
    assert counts.sum() == rows
    return counts


def topk_routing(tokens: int = 32768, top_k: int = 8, experts: int = EXPERTS, s: float = 1.2, seed: int = 6):
    """Per-token expert choices in the router-replay form: ``top_k`` distinct expert
    ids per token, experts drawn with Zipf(s) popularity over a seeded order
    (Gumbel top-k sampling without replacement), and positive routing weights
    normalised to sum 1 per token.

    Returns (ids int32 [tokens, top_k], weights float32 [tokens, top_k])."""
    rng = np.random.default_rng(seed)
    order = rng.permutation(experts)
    logp = np.empty(experts)
    logp[order] = -s * np.log(np.arange(1, experts + 1, dtype=np.float64))
    ids = np.empty((tokens, top_k), np.int32)
    step = 8192
    for t0 in range(0, tokens, step):
        t1 = min(tokens, t0 + step)
        keys = logp[None, :] + rng.gumbel(size=(t1 - t0, experts))
        ids[t0:t1] = np.argsort(-keys, axis=1, kind="stable")[:, :top_k]
    w = rng.uniform(0.05, 1.0, size=(tokens, top_k))
    weights = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, weights


# -------------------------------------------------------------- numpy inputs --
def tiny(seed: int = 0):
    """One expert: X [128 x 256] ~ N(0,1) with 1% of entries x30; W [256 x 256] ~ N(0, 0.02^2).

    Returns (x_bits, w_bits) as uint16 bf16 bit patterns."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((128, 256), dtype=np.float32)
    n_out = (x.size * 1) // 100
    idx = rng.choice(x.size, size=n_out, replace=False)
    x.reshape(-1)[idx] *= np.float32(30.0)
    w = rng.standard_normal((256, 256), dtype=np.float32) * np.float32(0.02)
    return bf16_bits(x), bf16_bits(w)


def quantizer_batch(rows: int = 16384, cols: int = HIDDEN, seed: int = 1):
    """Heterogeneous batch: X ~ N(0,1), 0.1% of channels x50, 1% of rows x1e-3.

    Returns (x_bits, hot_channels, small_rows)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols), dtype=np.float32)
    hot = np.sort(rng.choice(cols, size=max(1, cols // 1000), replace=False))
    small = np.sort(rng.choice(rows, size=max(1, rows // 100), replace=False))
    x[:, hot] *= np.float32(50.0)
    x[small, :] *= np.float32(1e-3)
    return bf16_bits(x), hot, small


def normal_bits(shape, std: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


# -------------------------------------------------------------- torch inputs --
def torch_normal(shape, std: float, seed: int, device="cuda"):
    """bf16 tensor of N(0, std^2) draws made on ``device`` from a seeded generator."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, float(std), generator=gen)
    return t.to(torch.bfloat16)
