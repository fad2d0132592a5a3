"""Helpers shared by the GPU parity tests (marshalling and row gathering)."""

import numpy as np
import torch

from exact_attention_fattn_gb300 import attention as A


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_fwd(inp, causal, scale):
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    o, lse = A.fattn_fwd(q, k, v, causal=causal, scale=scale)
    status = A.fattn_check_status()
    assert status == 0, f"fattn status {status}"
    return o, lse


def gather_rows(x, rows):
    """x [B,H,N,...] (tensor or array), rows [B,H,R] -> [B,H,R,...] numpy."""
    a = to_np(x) if isinstance(x, torch.Tensor) else x
    r = rows.numpy() if isinstance(rows, torch.Tensor) else rows
    B, H = r.shape[:2]
    return np.stack([np.stack([a[b, h, r[b, h]] for h in range(H)]) for b in range(B)])
