"""Seeded synthetic inputs for the ZipCCL BF16 exponent-coding path.

Shared by the oracle tests, the GPU parity tests and the benchmark.  This
module holds none of the method's arithmetic: it only draws numbers (numpy
PCG64, one SeedSequence child per tensor or chunk), rounds fp32 to BF16 words
(round to nearest even, the usual fp32 -> bf16 cast) and lays out chunks.

Workloads stand in for the pages' training runs (Llama3-8B on TorchTitan,
Qwen3-MoE, a 64-GPU cluster), which need models, datasets and a cluster:
  - ``pr1``: 1,048,576 values from N(0, 0.02^2), one chunk; plus all 65,536
    BF16 bit patterns as a second input;
  - ``gradient``: a 67,108,864-value bucket from N(0, 1e-3^2) in 8 equal
    per-destination chunks, and 8 independently seeded peer tensors of
    8,388,608 values each for the reduce;
  - ``moe``: 16,384 tokens x 4,096 hidden from N(0, 1), 0.1% of entries replaced
    by 10 * Student-t(3); top-2 of 64 experts from U[0, 1) gate logits (ties to
    the lower expert id); dispatch buffer in expert order, one chunk per expert;
  - ``fsdp``: 4 Llama-3-8B-shaped layers (q/o 4096x4096, k/v 1024x4096,
    gate/up 14336x4096, down 4096x14336) from N(0, 0.02^2), each weight split
    into 8 row chunks (224 chunks, 872,415,232 values);
  - ``stress``: 256 chunks of 1,048,576 values, chunk c from N(0, sigma_c^2)
    with log10(sigma_c) ~ U(-6, 2), except chunks with c mod 16 == 15, which
    hold uniform random 16-bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload", "f32_to_bf16_bits", "gaussian_bf16", "pr1", "all_patterns", "gradient",
    "gradient_peers", "moe", "fsdp", "stress", "random_chunks", "WORKLOADS",
]


def _rng(seed: int, *idx: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), *[int(i) for i in idx]]))


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """fp32 -> BF16 bit patterns (uint16), round to nearest even; NaN -> 0x7FC0."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    out = ((u + r) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def gaussian_bf16(n: int, sigma: float, seed: int, *idx: int, block: int = 1 << 24) -> np.ndarray:
    """n BF16 words drawn from N(0, sigma^2) (fp32 draw, then RNE to BF16)."""
    out = np.empty(int(n), dtype=np.uint16)
    rng = _rng(seed, *idx)
    for s in range(0, int(n), block):
        m = min(block, int(n) - s)
        z = rng.standard_normal(m, dtype=np.float32)
        z *= np.float32(sigma)
        out[s:s + m] = f32_to_bf16_bits(z)
    return out


@dataclass
class Workload:
    name: str
    x: np.ndarray                       # uint16 BF16 words, all chunks back to back
    chunk_elems: list[int]
    sigma: list[float] = field(default_factory=list)   # generating sigma per chunk (context only)
    note: str = ""

    @property
    def n(self) -> int:
        return int(self.x.size)


def pr1(seed: int = 1) -> Workload:
    n = 1_048_576
    return Workload("pr1", gaussian_bf16(n, 0.02, seed, 0), [n], [0.02],
                    "1,048,576 x N(0, 0.02^2), one chunk")


def all_patterns() -> Workload:
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return Workload("all_patterns", x, [65536], [], "every BF16 bit pattern 0..65535 in order")


def gradient(seed: int = 100, n: int = 67_108_864, ranks: int = 8) -> Workload:
    per = n // ranks
    x = np.concatenate([gaussian_bf16(per, 1e-3, seed, r) for r in range(ranks)])
    return Workload("gradient", x, [per] * ranks, [1e-3] * ranks,
                    f"{n:,} x N(0, 1e-3^2) in {ranks} per-destination chunks")


def gradient_peers(seed: int = 100, per: int = 8_388_608, k: int = 8) -> list[np.ndarray]:
    """k independently seeded peer tensors (the chunk each peer sends to this rank)."""
    return [gaussian_bf16(per, 1e-3, seed, 1000 + p) for p in range(k)]


def moe(seed: int = 200, tokens: int = 16_384, hidden: int = 4_096, experts: int = 64,
        top_k: int = 2, outlier_frac: float = 1e-3) -> Workload:
    rng = _rng(seed, 0)
    X = rng.standard_normal((tokens, hidden), dtype=np.float32)
    n_out = int(round(outlier_frac * X.size))
    pos = rng.choice(X.size, size=n_out, replace=False)
    X.reshape(-1)[pos] = (10.0 * rng.standard_t(3, size=n_out)).astype(np.float32)
    logits = rng.random((tokens, experts), dtype=np.float32)
    # top-k per token; ties broken toward the lower expert id (stable sort on -logit)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :top_k]
    tok = np.repeat(np.arange(tokens), top_k)
    exp_ids = order.reshape(-1)
    perm = np.lexsort((tok, exp_ids))      # expert-major, token order inside an expert
    rows = tok[perm]
    counts = np.bincount(exp_ids, minlength=experts)
    Xb = f32_to_bf16_bits(X.reshape(-1)).reshape(tokens, hidden)
    buf = Xb[rows].reshape(-1)
    return Workload("moe", buf, [int(c) * hidden for c in counts], [1.0] * experts,
                    f"{tokens}x{hidden} N(0,1) + {n_out} 10*t3 outliers, top-{top_k} of {experts} "
                    f"experts -> {rows.size} dispatch rows")


FSDP_SHAPES = [("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
               ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336)]


def fsdp(seed: int = 300, layers: int = 4, shards: int = 8) -> Workload:
    total = sum(r * c for _, r, c in FSDP_SHAPES) * layers
    x = np.empty(total, dtype=np.uint16)
    chunks, pos = [], 0
    for layer in range(layers):
        for wi, (_, rows, cols) in enumerate(FSDP_SHAPES):
            m = rows * cols
            x[pos:pos + m] = gaussian_bf16(m, 0.02, seed, layer, wi)
            pos += m
            chunks += [(rows // shards) * cols] * shards
    return Workload("fsdp", x, chunks, [0.02] * len(chunks),
                    f"{layers} Llama-3-8B-shaped layers, N(0, 0.02^2), {len(chunks)} row chunks")


def stress(seed: int = 400, chunks: int = 256, per: int = 1_048_576) -> Workload:
    rng = _rng(seed, 0)
    log_sig = rng.uniform(-6.0, 2.0, size=chunks)
    parts, sig = [], []
    for c in range(chunks):
        if c % 16 == 15:
            parts.append(_rng(seed, 1, c).integers(0, 65536, size=per, dtype=np.uint16))
            sig.append(float("nan"))
        else:
            s = float(10.0 ** log_sig[c])
            parts.append(gaussian_bf16(per, s, seed, 2, c))
            sig.append(s)
    return Workload("stress", np.concatenate(parts), [per] * chunks, sig,
                    f"{chunks} x {per:,}; sigma log-uniform on [1e-6, 1e2]; every 16th chunk uniform u16")


def random_chunks(seed: int, n_chunks: int, max_elems: int, sigma_range=(1e-4, 10.0),
                  empty_prob: float = 0.1) -> Workload:
    """Small seeded mixes: ragged chunk sizes, empty chunks, mixed scales and specials."""
    rng = _rng(seed, 0)
    sizes = [0 if rng.random() < empty_prob else int(rng.integers(1, max_elems + 1)) for _ in range(n_chunks)]
    parts, sig = [], []
    for c, m in enumerate(sizes):
        s = float(np.exp(rng.uniform(np.log(sigma_range[0]), np.log(sigma_range[1]))))
        g = gaussian_bf16(m, s, seed, 1, c)
        if m and rng.random() < 0.3:      # sprinkle zeros / specials / random patterns
            k = max(1, m // 50)
            idx = rng.integers(0, m, size=k)
            g[idx] = rng.integers(0, 65536, size=k, dtype=np.uint16)
        parts.append(g)
        sig.append(s)
    x = np.concatenate(parts) if parts else np.zeros(0, dtype=np.uint16)
    return Workload(f"random{seed}", x, sizes, sig, "ragged seeded mix")


WORKLOADS = {"pr1": pr1, "gradient": gradient, "moe": moe, "fsdp": fsdp, "stress": stress}
