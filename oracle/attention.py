"""Oracle: fp64 masked softmax attention, forward and backward, on the CPU.

Test infrastructure only (see the package header).

What it computes (CompileMask section 3.3.2: invisible scores are replaced with -inf before the
softmax, so descriptor-guided attention equals softmax attention under the dense mask):

  s      = scale * q k^T,  s[i, j] = -inf where (i, j) is not visible
  lse_i  = log sum_j exp(s[i, j])                  (natural log; -inf for a row that sees nothing)
  p      = exp(s - lse)                            (0 on a row that sees nothing)
  o      = p v
  dv     = p^T do,  dp = do v^T,  D_i = sum_j p[i, j] dp[i, j]
  ds     = p * (dp - D),  dq = scale * ds k,  dk = scale * ds^T q

Readings: scale = 1/sqrt(d); the LSE is reported in natural log.  Inputs are the bf16 values
widened to fp64.  Rows are independent in the forward pass, so the functions may walk the query
rows in blocks (``block_rows``) to bound memory at 32K; dk and dv are sums over rows.
"""
from __future__ import annotations

import math
from typing import Callable

import torch

MaskRows = Callable[[int, int], "object"]  # (row0, row1) -> bool array/tensor [row1-row0, S]


def _as64(x) -> torch.Tensor:
    return x.to(torch.float64) if isinstance(x, torch.Tensor) else torch.as_tensor(x, dtype=torch.float64)


def _mask_block(mask, r0: int, r1: int) -> torch.Tensor:
    m = mask(r0, r1) if callable(mask) else mask[r0:r1]
    return torch.as_tensor(m, dtype=torch.bool)


def attention_forward(q, k, v, mask, scale: float | None = None,
                      block_rows: int | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """o [S, d] fp64 and lse [S] fp64 for one (batch, head).

    ``mask`` is a bool [S, S] array or a callable returning rows [r0, r1) of it.
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    S, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    br = S if block_rows is None else block_rows
    o = torch.zeros(S, v.shape[1], dtype=torch.float64)
    lse = torch.empty(S, dtype=torch.float64)
    for r0 in range(0, S, br):
        r1 = min(S, r0 + br)
        s = scale * (q[r0:r1] @ k.T)
        s = s.masked_fill(~_mask_block(mask, r0, r1), float("-inf"))
        l = torch.logsumexp(s, dim=1)
        seen = torch.isfinite(l)
        p = torch.where(seen[:, None], torch.exp(s - l[:, None]), torch.zeros_like(s))
        o[r0:r1] = p @ v
        lse[r0:r1] = l
    return o, lse


def attention_backward(q, k, v, do, mask, scale: float | None = None,
                       block_rows: int | None = None) -> tuple[torch.Tensor, ...]:
    """dq, dk, dv [S, d] fp64 for one (batch, head), recomputing p from the definition."""
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    S, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    br = S if block_rows is None else block_rows
    dq = torch.zeros_like(q)
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    for r0 in range(0, S, br):
        r1 = min(S, r0 + br)
        s = scale * (q[r0:r1] @ k.T)
        s = s.masked_fill(~_mask_block(mask, r0, r1), float("-inf"))
        l = torch.logsumexp(s, dim=1)
        seen = torch.isfinite(l)
        p = torch.where(seen[:, None], torch.exp(s - l[:, None]), torch.zeros_like(s))
        dv += p.T @ do[r0:r1]
        dp = do[r0:r1] @ v.T
        D = (p * dp).sum(dim=1)
        ds = p * (dp - D[:, None])
        dq[r0:r1] = scale * (ds @ k)
        dk += scale * (ds.T @ q[r0:r1])
    return dq, dk, dv
