"""Seeded synthetic inputs for the BackLite attention workloads.

This module only draws random numbers and arranges them into tensors; it
holds none of the attention arithmetic.  Both the CUDA path (tests, bench)
and the CPU oracle read their inputs from here, so the two sides always see
the same bf16 values.

Recipe (one numpy PCG64 stream per call, seed 0 unless stated):

* ``iid``: Q, K, V and G_O are independent N(0, 1).
* ``clustered``: each token t belongs to a cluster c(t).  Per (batch,
  kv head) a centre mu_c ~ N(0, I_d) is drawn for every cluster; every query
  head of that kv head's group sees the same centres.  Then
  Q[b,t,h] = alpha*mu_{c(t)} + N(0,1) and K[b,t,hk] = alpha*mu_{c(t)} + N(0,1)
  with independent noise, and V, G_O ~ N(0,1).  For the 1-D runs
  c(t) = floor(t / run) mod C; for the video-shaped grid the tokens of a
  T x Y x X latent grid are flattened t-major and c(t) is the index of the
  3-D patch that holds the token.

Values are drawn in fp32 and rounded to bf16 (round to nearest even); the
oracle reads exactly these bf16 values, widened to fp64.

The workloads mirror the shapes that the BackLite pages motivate: the
long-sequence video DiT regime ("Introducing BackLite", Introduction: 32k
tokens for a 5 s 480p Wan 2.1 video) and long-context LLM training (same
section: 128k contexts), causal and sliding-window LLM training (same
post, Training Nanochat: windows of 1024 and 2048), plus two small cases and
a GQA case ("BackLite" README, Forward signature: key/value carry
``heads_k`` heads).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    n: int
    H: int
    Hk: int
    d: int
    block_q: int
    block_k: int
    negl_probs: tuple
    kind: str                      # "iid" | "runs" | "grid"
    alpha: float = 0.0
    run: int = 0
    clusters: int = 0
    grid: tuple = ()               # (T, Y, X) for kind == "grid"
    patch: tuple = ()              # (pt, py, px) for kind == "grid"
    causal: bool = False           # query r attends keys c <= r
    window: int = 0                # with causal: keys r - window < c <= r

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def T_r(self) -> int:
        return -(-self.n // self.block_q)

    @property
    def T_c(self) -> int:
        return -(-self.n // self.block_k)

    def attending_pairs(self) -> int:
        """(query, key) pairs per head that attend under causal / window."""
        n = self.n
        if not self.causal:
            return n * n
        if not self.window or self.window >= n:
            return n * (n + 1) // 2
        w = self.window
        return w * (w + 1) // 2 + (n - w) * w

    def dense_bwd_flop(self) -> float:
        """10*B*H*pairs*d: the five contractions of the dense backward over the
        (query, key) pairs that attend (n^2 without causal structure)."""
        return 10.0 * self.B * self.H * self.attending_pairs() * self.d

    def dense_fwd_flop(self) -> float:
        return 4.0 * self.B * self.H * self.attending_pairs() * self.d


WORKLOADS = {
    "tiny_n256_d64": Workload("tiny_n256_d64", B=1, n=256, H=1, Hk=1, d=64,
                              block_q=64, block_k=64, negl_probs=(0.0, 0.05),
                              kind="iid"),
    "clustered_n4096_d64": Workload("clustered_n4096_d64", B=2, n=4096, H=12, Hk=12,
                                    d=64, block_q=128, block_k=128,
                                    negl_probs=(0.05,), kind="runs", alpha=3.0,
                                    run=64, clusters=32),
    "gqa_n8192_d128": Workload("gqa_n8192_d128", B=1, n=8192, H=32, Hk=8, d=128,
                               block_q=128, block_k=128,
                               negl_probs=(0.01, 0.05, 0.1), kind="runs",
                               alpha=2.5, run=64, clusters=64),
    "video_n32760_d128": Workload("video_n32760_d128", B=1, n=32760, H=40, Hk=40,
                                  d=128, block_q=128, block_k=128,
                                  negl_probs=(0.05,), kind="grid", alpha=3.0,
                                  grid=(21, 30, 52), patch=(3, 6, 8)),
    # the video grid with 8 heads: same per-head structure, a small case for profiling
    "video_n32760_d128_h8": Workload("video_n32760_d128_h8", B=1, n=32760, H=8, Hk=8,
                                     d=128, block_q=128, block_k=128,
                                     negl_probs=(0.05,), kind="grid", alpha=3.0,
                                     grid=(21, 30, 52), patch=(3, 6, 8)),
    "long_n131072_d128": Workload("long_n131072_d128", B=1, n=131072, H=32, Hk=8,
                                  d=128, block_q=128, block_k=128,
                                  negl_probs=(0.05,), kind="runs", alpha=3.0,
                                  run=128, clusters=256),
    # decoder-style LLM training: causal, and causal with the 1024 / 2048
    # sliding windows of the BackLite blog's Nanochat runs
    "llm_causal_n16384_d128": Workload("llm_causal_n16384_d128", B=1, n=16384, H=32, Hk=8,
                                       d=128, block_q=128, block_k=128,
                                       negl_probs=(0.05,), kind="runs", alpha=3.0,
                                       run=64, clusters=64, causal=True),
    "llm_window2048_n16384_d128": Workload("llm_window2048_n16384_d128", B=1, n=16384, H=32,
                                           Hk=8, d=128, block_q=128, block_k=128,
                                           negl_probs=(0.05,), kind="runs", alpha=3.0,
                                           run=64, clusters=64, causal=True, window=2048),
}


def custom(name="custom", *, B, n, H, Hk, d, block_q=128, block_k=128,
           kind="runs", alpha=3.0, run=64, clusters=16, negl_probs=(0.05,),
           causal=False, window=0):
    """A workload of arbitrary shape with the 1-D clustered (or iid) recipe."""
    return Workload(name, B=B, n=n, H=H, Hk=Hk, d=d, block_q=block_q,
                    block_k=block_k, negl_probs=tuple(negl_probs), kind=kind,
                    alpha=alpha, run=run, clusters=clusters, causal=causal,
                    window=window)


def cluster_of_token(w: Workload) -> np.ndarray:
    """Cluster index c(t) for every token t (int64, length n)."""
    t = np.arange(w.n, dtype=np.int64)
    if w.kind == "runs":
        return (t // w.run) % w.clusters
    if w.kind == "grid":
        T, Y, X = w.grid
        assert T * Y * X == w.n
        pt, py, px = w.patch
        ny, nx = -(-Y // py), -(-X // px)
        tt, rem = t // (Y * X), t % (Y * X)
        yy, xx = rem // X, rem % X
        return (tt // pt) * (ny * nx) + (yy // py) * nx + (xx // px)
    raise ValueError(w.kind)


def n_clusters(w: Workload) -> int:
    if w.kind == "runs":
        return w.clusters
    if w.kind == "grid":
        T, Y, X = w.grid
        pt, py, px = w.patch
        return (-(-T // pt)) * (-(-Y // py)) * (-(-X // px))
    return 0


def _to_bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(x).to(torch.bfloat16)


def generate(w: Workload, seed: int = 0, with_grad_out: bool = True):
    """Draw (q, k, v, g_o) for a workload as CPU bf16 tensors in BSHD layout.

    q, g_o: [B, n, H, d]; k, v: [B, n, Hk, d].  Deterministic in ``seed``.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    B, n, H, Hk, d = w.B, w.n, w.H, w.Hk, w.d
    G = H // Hk
    f32 = np.float32
    if w.kind == "iid":
        q = rng.standard_normal((B, n, H, d), dtype=f32)
        k = rng.standard_normal((B, n, Hk, d), dtype=f32)
    else:
        C = n_clusters(w)
        mu = rng.standard_normal((B, Hk, C, d), dtype=f32)
        c = cluster_of_token(w)
        # centre of every token for every (batch, kv head): [B, n, Hk, d]
        centre = np.ascontiguousarray(
            np.transpose(mu[:, :, c, :], (0, 2, 1, 3))) * f32(w.alpha)
        q = rng.standard_normal((B, n, H, d), dtype=f32)
        q = q.reshape(B, n, Hk, G, d)
        q += centre[:, :, :, None, :]
        q = q.reshape(B, n, H, d)
        k = rng.standard_normal((B, n, Hk, d), dtype=f32)
        k += centre
        del centre
    v = rng.standard_normal((B, n, Hk, d), dtype=f32)
    out = [_to_bf16(q), _to_bf16(k), _to_bf16(v)]
    del q, k, v
    if with_grad_out:
        out.append(_to_bf16(rng.standard_normal((B, n, H, d), dtype=f32)))
    else:
        out.append(None)
    return tuple(out)


def generate_packed(w: Workload, lengths, seed: int = 0):
    """A packed variable-length batch: sequence s of ``lengths`` is drawn as the
    workload ``w`` with B = 1 and n = lengths[s] (seed ``seed + s``), and the
    sequences are stacked along the token axis.  Returns (cu_seqlens, q, k, v,
    g_o) with q, g_o [total, H, d] and k, v [total, Hk, d] CPU bf16 tensors;
    empty sequences own no rows."""
    cu = [0]
    parts = []
    for s, n in enumerate(lengths):
        cu.append(cu[-1] + int(n))
        if n:
            ws = dataclasses.replace(w, B=1, n=int(n))
            parts.append([x[0] for x in generate(ws, seed=seed + s)])
    q, k, v, go = (torch.cat([p[i] for p in parts], dim=0).contiguous() for i in range(4))
    return cu, q, k, v, go


def document_lengths(total: int, seed: int = 0, median: int = 1536, sigma: float = 1.0,
                     lo: int = 64, hi: int = 8192):
    """Lengths of documents packed into one batch of ``total`` tokens: log-normal
    draws (median ``median``, shape ``sigma``) clipped to [lo, hi], the last
    one cut so that the lengths add up to ``total``."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    left = total
    while left > 0:
        n = int(np.clip(round(median * math.exp(sigma * rng.standard_normal())), lo, hi))
        n = min(n, left)
        out.append(n)
        left -= n
    return out


@dataclasses.dataclass(frozen=True)
class Packed:
    """A packed variable-length batch: the per-sequence recipe of ``base`` (its
    B and n are ignored) and the sequence lengths."""
    name: str
    base: Workload
    lengths: tuple

    @property
    def total(self) -> int:
        return sum(self.lengths)

    def seq(self, n: int) -> Workload:
        return dataclasses.replace(self.base, B=1, n=n)

    def dense_fwd_flop(self) -> float:
        return sum(self.seq(n).dense_fwd_flop() for n in self.lengths if n)

    def dense_bwd_flop(self) -> float:
        return sum(self.seq(n).dense_bwd_flop() for n in self.lengths if n)


PACKED = {
    # decoder pre-training batch: 16384 tokens of documents of mixed length
    "llm_packed_causal_t16384_d128": Packed(
        "llm_packed_causal_t16384_d128",
        Workload("doc", B=1, n=1, H=32, Hk=8, d=128, block_q=128, block_k=128,
                 negl_probs=(0.05,), kind="runs", alpha=3.0, run=64, clusters=64,
                 causal=True),
        tuple(document_lengths(16384, seed=0))),
    # four equal video clips of the 32760-token grid's 1-D stand-in: one launch group
    "video_packed_4x8190_d128": Packed(
        "video_packed_4x8190_d128",
        Workload("clip", B=1, n=1, H=40, Hk=40, d=128, block_q=128, block_k=128,
                 negl_probs=(0.05,), kind="runs", alpha=3.0, run=128, clusters=64),
        (8190, 8190, 8190, 8190)),
}
