"""Seeded synthetic inputs for the five mask workloads.

This module only draws random numbers: segment lengths (the per-batch metadata) and bf16
Q/K/V/dO tensors.  It holds none of the masking or attention arithmetic, so the CPU oracle and
the CUDA path can both take their inputs from it without sharing any of the method.

Workloads (sizes follow the CompileMask evaluation, section 4.1 "Experimental Setup": causal,
shared-prompt reward model, HSTU and multi-interval masks up to 32K; the recommendation data set
used there is not available, so every length is drawn here instead):

  1 packed-document causal   B=1  H=2  S=512    d=64   three documents, each >= 32 tokens
  2 plain causal             B=2  H=16 S=8192   d=128  one segment
  3 shared-prompt RM         B=1  H=32 S=32768  d=128  prompt P ~ U[S/8, 3S/8], then 4 responses
  4 HSTU                     B=4  H=16 S=16384  d=128  history h ~ U[S/2, S - S/16] per sample
  5 three-interval packed    B=2  H=32 S=32768  d=128  prefix S/64, documents ~ U[S/32, 3S/16]
  6 varlen packed HSTU       B=2  H=16 S=32768  d=128  users of length ~ U[S/32, S/4] packed to S,
                                                     each a history (50-90 %) then candidates

Metadata layout: ``seg`` is int32 [B, nseg_max + 1] with seg[b, 0] = 0 and seg[b, nseg[b]] = S,
entries past nseg[b] repeat S; ``nseg`` is int32 [B].
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    id: int
    name: str
    B: int
    H: int
    S: int
    d: int


WORKLOADS = {
    1: Workload(1, "packed_doc_causal_512", 1, 2, 512, 64),
    2: Workload(2, "causal_8k", 2, 16, 8192, 128),
    3: Workload(3, "shared_prompt_rm_32k", 1, 32, 32768, 128),
    4: Workload(4, "hstu_16k", 4, 16, 16384, 128),
    5: Workload(5, "three_interval_packed_32k", 2, 32, 32768, 128),
    6: Workload(6, "varlen_hstu_packed_32k", 2, 16, 32768, 128),
}


def scaled(w: Workload, S: int, B: int | None = None, H: int | None = None,
           d: int | None = None) -> Workload:
    """The same mask family at another size (used for small parity cases)."""
    return Workload(w.id, f"{w.name}@S{S}", B or w.B, H or w.H, S, d or w.d)


def _lengths_to_seg(lengths_per_batch: list[list[int]], S: int) -> tuple[np.ndarray, np.ndarray]:
    nseg = np.array([len(l) for l in lengths_per_batch], dtype=np.int32)
    width = int(nseg.max()) + 1
    seg = np.full((len(lengths_per_batch), width), S, dtype=np.int32)
    for b, lens in enumerate(lengths_per_batch):
        pos = 0
        seg[b, 0] = 0
        for k, n in enumerate(lens):
            pos += int(n)
            seg[b, k + 1] = pos
        assert pos == S, (pos, S)
    return seg, nseg


def segments(wid: int, B: int, S: int, seed: int | None = None) -> tuple[np.ndarray, np.ndarray]:
    """Draw the segment boundaries of workload family ``wid`` for B samples of length S."""
    rng = np.random.default_rng(1000 + wid if seed is None else seed)
    out: list[list[int]] = []
    for _ in range(B):
        if wid == 1:
            # three documents, each at least 32 long (S/16 when S is small)
            m = min(32, S // 16)
            lens = (m + rng.multinomial(S - 3 * m, [1 / 3] * 3)).tolist()
        elif wid == 2:
            lens = [S]
        elif wid == 3:
            while True:
                P = int(rng.integers(S // 8, 3 * S // 8, endpoint=True))
                resp = rng.multinomial(S - P, [1 / 4] * 4)
                if (resp > 0).all():
                    break
            lens = [P] + resp.tolist()
        elif wid == 4:
            h = int(rng.integers(S // 2, S - S // 16, endpoint=True))
            lens = [h, S - h]
        elif wid == 5:
            b = S // 64
            lens = [b]
            total = b
            while total < S:
                n = int(rng.integers(S // 32, 3 * S // 16, endpoint=True))
                n = min(n, S - total)
                lens.append(n)
                total += n
        elif wid == 6:
            # users packed back to back (variable lengths, as in a batch of recommendation
            # sequences); the last one takes the remainder, or joins the previous user when the
            # remainder is too short; each user splits into history and candidates
            lo, hi = max(4, S // 32), max(8, S // 4)
            users: list[int] = []
            total = 0
            while total < S:
                n = int(rng.integers(lo, hi, endpoint=True))
                n = min(n, S - total)
                if n < max(4, S // 128) and users:
                    users[-1] += n
                else:
                    users.append(n)
                total += n
            lens = []
            for n in users:
                h = int(np.floor(n * rng.uniform(0.5, 0.9)))
                h = min(max(h, 1), n - 1)
                lens += [h, n - h]
        else:
            raise ValueError(f"unknown workload {wid}")
        out.append([int(x) for x in lens])
    return _lengths_to_seg(out, S)


def random_segments(B: int, S: int, max_segs: int, seed: int, min_len: int = 1):
    """Arbitrary segmentations (for randomized descriptor checks): 1..max_segs segments."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(B):
        n = int(rng.integers(1, max_segs, endpoint=True))
        n = max(1, min(n, S // max(min_len, 1)))
        cuts = np.sort(rng.choice(np.arange(1, S), size=n - 1, replace=False)) if n > 1 else []
        bounds = [0] + [int(c) for c in cuts] + [S]
        out.append([bounds[k + 1] - bounds[k] for k in range(n)])
    return _lengths_to_seg(out, S)


def head_tensors(wid: int, b: int, h: int, S: int, d: int, H: int,
                 seed: int | None = None) -> tuple[torch.Tensor, ...]:
    """Q, K, V, dO of one (batch, head): fp32 N(0,1) rounded to bf16, each [S, d].

    Every head has its own generator so that one head can be regenerated without the others.
    """
    base = (2000 + wid) if seed is None else seed
    g = torch.Generator(device="cpu")
    g.manual_seed(base * 1_000_003 + (b * H + h))
    return tuple(torch.randn(S, d, generator=g, dtype=torch.float32).to(torch.bfloat16)
                 for _ in range(4))


def full_tensors(w: Workload, seed: int | None = None, heads=None) -> tuple[torch.Tensor, ...]:
    """Q, K, V, dO as bf16 [B, H, S, d] on the CPU (pinned-free, contiguous)."""
    Q, K, V, dO = (torch.empty(w.B, w.H, w.S, w.d, dtype=torch.bfloat16) for _ in range(4))
    for b in range(w.B):
        for h in range(w.H):
            q, k, v, do = head_tensors(w.id, b, h, w.S, w.d, w.H, seed)
            Q[b, h], K[b, h], V[b, h], dO[b, h] = q, k, v, do
    return Q, K, V, dO
