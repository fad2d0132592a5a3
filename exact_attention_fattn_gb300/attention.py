"""Python entry points over libfattn, with the C ABI's names.

PyTorch provides device memory and streams only: outputs are allocated as
torch tensors and their raw pointers, with the current CUDA stream, are
handed to the library.  Nothing here computes attention.
"""

from __future__ import annotations

import math

import torch

from . import _lib


def _stream_ptr(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check_inputs(tensors, d_expected=None):
    t0 = tensors[0]
    if not t0.is_cuda:
        raise ValueError("libfattn works on CUDA tensors; move the inputs to the GPU first")
    for t in tensors:
        if t.dtype != torch.bfloat16:
            raise TypeError(f"expected bfloat16 tensors, got {t.dtype}")
        if t.dim() != 4 or t.shape != t0.shape:
            raise ValueError("q, k, v (and o, dO) must share one [B, H, N, d] shape")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous [B, H, N, d]")
        if t.device != t0.device:
            raise ValueError("tensors must be on one device")


def _check_out(t, shape, dtype, device, name):
    """A caller-provided output buffer must be exactly what the kernel writes."""
    if (t.dtype != dtype or tuple(t.shape) != tuple(shape) or t.device != device
            or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} "
                         f"on {device}")
    return t


def default_scale(d: int) -> float:
    """1/sqrt(d) ("6.1 FlashAttention V1详解" §1.1), as an fp32 value."""
    return float(torch.tensor(1.0 / math.sqrt(d), dtype=torch.float32))


def fattn_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None):
    """Forward pass; returns (O bf16 [B,H,N,d], L fp32 [B,H,N])."""
    _check_inputs([q, k, v])
    B, H, N, d = q.shape
    scale = default_scale(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else _check_out(out, q.shape, q.dtype, q.device, "out")
    l = (torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None
         else _check_out(lse, (B, H, N), torch.float32, q.device, "lse"))
    lib = _lib.load()
    with torch.cuda.device(q.device):
        rc = lib.fattn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                           B, H, N, d, int(bool(causal)), scale, _stream_ptr(q.device))
    _lib.check("fattn_fwd", rc)
    return o, l


def fattn_quantize_fp8(x, transposed: bool = False, signs=None):
    """Block-quantize a bf16 [B,H,N,d] tensor (d = 128) to e4m3 codes.

    Returns (codes, scales): uint8 [B,H,N,d] (or [B,H,d,Np] when
    ``transposed``, Np = N rounded up to 128) and fp32 [B,H,ceil(N/128)].
    With ``signs`` (fp32 CUDA tensor [d] of +-1) the rows are first rotated
    by diag(signs) H / sqrt(d) (incoherent processing; for Q and K only).
    """
    _check_inputs([x])
    B, H, N, d = x.shape
    lib = _lib.load()
    if signs is not None:
        if transposed:
            raise ValueError("the rotation applies to Q and K, which are not transposed")
        if (signs.dtype != torch.float32 or signs.device != x.device or signs.numel() != d
                or not signs.is_contiguous()):
            raise TypeError("signs must be a contiguous fp32 tensor of d values on x's device")
        if d != 128:
            raise ValueError("the FP8 path supports d = 128 only")
        codes = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device)
        scales = torch.empty((B, H, (N + 127) // 128), dtype=torch.float32, device=x.device)
        with torch.cuda.device(x.device):
            rc = lib.fattn_quantize_fp8_rotated(x.data_ptr(), signs.data_ptr(), codes.data_ptr(),
                                                scales.data_ptr(), B, H, N, d,
                                                _stream_ptr(x.device))
        _lib.check("fattn_quantize_fp8_rotated", rc)
        return codes, scales
    nbytes = int(lib.fattn_fp8_codes_bytes(B, H, N, d, int(bool(transposed))))
    if nbytes == 0:
        raise ValueError("the FP8 path supports d = 128 only")
    np_ = (N + 127) // 128 * 128
    shape = (B, H, d, np_) if transposed else (B, H, N, d)
    codes = torch.empty(shape, dtype=torch.uint8, device=x.device)
    scales = torch.empty((B, H, (N + 127) // 128), dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        rc = lib.fattn_quantize_fp8(x.data_ptr(), codes.data_ptr(), scales.data_ptr(), B, H, N, d,
                                    int(bool(transposed)), _stream_ptr(x.device))
    _lib.check("fattn_quantize_fp8", rc)
    return codes, scales


def fattn_fwd_fp8(q8, sq, k8, sk, v8t, sv, causal: bool = False, scale: float | None = None,
                  out=None, lse=None):
    """FP8 forward on block-quantized inputs (from fattn_quantize_fp8; V
    transposed); returns (O bf16 [B,H,N,d], L fp32 [B,H,N])."""
    for t in (q8, k8, v8t):
        if t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous():
            raise TypeError("q8, k8, v8t must be contiguous uint8 CUDA tensors")
    for t in (sq, sk, sv):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise TypeError("scales must be contiguous fp32 tensors")
    if any(t.device != q8.device for t in (k8, v8t, sq, sk, sv)):
        raise ValueError("codes and scales must be on one CUDA device")
    B, H, N, d = q8.shape
    if k8.shape != q8.shape or v8t.shape[:3] != (B, H, d):
        raise ValueError("q8, k8 must be [B,H,N,d] and v8t [B,H,d,Np]")
    nt = (N + 127) // 128
    if any(t.shape != (B, H, nt) for t in (sq, sk, sv)):
        raise ValueError("scales must be [B,H,ceil(N/128)] fp32 (one per 128-row block)")
    scale = default_scale(d) if scale is None else float(scale)
    o = (torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if out is None
         else _check_out(out, (B, H, N, d), torch.bfloat16, q8.device, "out"))
    l = (torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None
         else _check_out(lse, (B, H, N), torch.float32, q8.device, "lse"))
    lib = _lib.load()
    with torch.cuda.device(q8.device):
        rc = lib.fattn_fwd_fp8(q8.data_ptr(), sq.data_ptr(), k8.data_ptr(), sk.data_ptr(),
                               v8t.data_ptr(), sv.data_ptr(), o.data_ptr(), l.data_ptr(),
                               B, H, N, d, int(bool(causal)), scale, _stream_ptr(q8.device))
    _lib.check("fattn_fwd_fp8", rc)
    return o, l


def fattn_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(_lib.load().fattn_bwd_workspace_bytes(B, H, N, d))


def workspace_for(q) -> torch.Tensor:
    """A caller-owned uint8 workspace of the size fattn_bwd needs."""
    B, H, N, d = q.shape
    nbytes = fattn_bwd_workspace_bytes(B, H, N, d)
    if nbytes == 0:
        raise ValueError("unsupported shape")
    return torch.empty(nbytes, dtype=torch.uint8, device=q.device)


def _check_workspace(ws, q):
    if ws.dtype != torch.uint8 or ws.device != q.device or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 tensor on the inputs' device")
    return ws   # its size is checked by the library


def fattn_bwd(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None,
              workspace=None, dq=None, dk=None, dv=None):
    """Backward pass; returns (dQ, dK, dV), bf16 [B,H,N,d]."""
    _check_inputs([q, k, v, o, do])
    B, H, N, d = q.shape
    _check_out(lse, (B, H, N), torch.float32, q.device, "lse")
    scale = default_scale(d) if scale is None else float(scale)
    ws = workspace_for(q) if workspace is None else _check_workspace(workspace, q)
    dq = torch.empty_like(q) if dq is None else _check_out(dq, q.shape, q.dtype, q.device, "dq")
    dk = torch.empty_like(k) if dk is None else _check_out(dk, q.shape, q.dtype, q.device, "dk")
    dv = torch.empty_like(v) if dv is None else _check_out(dv, q.shape, q.dtype, q.device, "dv")
    lib = _lib.load()
    with torch.cuda.device(q.device):
        rc = lib.fattn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                           lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                           ws.data_ptr(), ws.numel(), B, H, N, d, int(bool(causal)), scale,
                           _stream_ptr(q.device))
    _lib.check("fattn_bwd", rc)
    return dq, dk, dv


def fattn_bwd_prepare(o, do, lse, workspace):
    _check_inputs([o, do])
    B, H, N, d = o.shape
    _check_out(lse, (B, H, N), torch.float32, o.device, "lse")
    _check_workspace(workspace, o)
    lib = _lib.load()
    with torch.cuda.device(o.device):
        rc = lib.fattn_bwd_prepare(o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                                   workspace.data_ptr(), workspace.numel(), B, H, N, d,
                                   _stream_ptr(o.device))
    _lib.check("fattn_bwd_prepare", rc)


def fattn_bwd_main(q, k, v, do, workspace, dk, dv, causal: bool = False,
                   scale: float | None = None):
    _check_inputs([q, k, v, do, dk, dv])
    _check_workspace(workspace, q)
    B, H, N, d = q.shape
    scale = default_scale(d) if scale is None else float(scale)
    lib = _lib.load()
    with torch.cuda.device(q.device):
        rc = lib.fattn_bwd_main(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                                workspace.data_ptr(), workspace.numel(), dk.data_ptr(),
                                dv.data_ptr(), B, H, N, d, int(bool(causal)), scale,
                                _stream_ptr(q.device))
    _lib.check("fattn_bwd_main", rc)


def fattn_bwd_finish(workspace, dq, scale: float | None = None):
    _check_inputs([dq])
    _check_workspace(workspace, dq)
    B, H, N, d = dq.shape
    scale = default_scale(d) if scale is None else float(scale)
    lib = _lib.load()
    with torch.cuda.device(dq.device):
        rc = lib.fattn_bwd_finish(workspace.data_ptr(), workspace.numel(), dq.data_ptr(),
                                  B, H, N, d, scale, _stream_ptr(dq.device))
    _lib.check("fattn_bwd_finish", rc)


def fattn_bwd_preprocess(o, do, D, dq_accum):
    _check_inputs([o, do])
    B, H, N, d = o.shape
    _check_out(D, (B, H, N), torch.float32, o.device, "D")
    _check_out(dq_accum, (B, H, N, d), torch.float32, o.device, "dq_accum")
    lib = _lib.load()
    with torch.cuda.device(o.device):
        rc = lib.fattn_bwd_preprocess(o.data_ptr(), do.data_ptr(), D.data_ptr(),
                                      dq_accum.data_ptr(), B, H, N, d, _stream_ptr(o.device))
    _lib.check("fattn_bwd_preprocess", rc)


def fattn_bwd_schedule(B: int, H: int, N: int, d: int, causal: bool, grid: int, l2_bytes: int,
                       deterministic: bool = False):
    """The backward kernel's static work schedule, computed on the host.

    Returns (item_cta, cta_q_tiles): int32 [B*H, ceil(N/128)] with the CTA
    that processes each K/V tile (-1 none, -2 several), and int64 [grid] with
    the Q tiles each CTA walks.  Needs no GPU.
    """
    n_tiles = (N + 127) // 128
    item_cta = torch.empty(B * H * n_tiles, dtype=torch.int32)
    cta_q_tiles = torch.empty(max(grid, 0), dtype=torch.int64)
    rc = _lib.load().fattn_bwd_schedule(B, H, N, d, int(bool(causal)), int(bool(deterministic)),
                                        grid, l2_bytes, item_cta.data_ptr(),
                                        cta_q_tiles.data_ptr())
    _lib.check("fattn_bwd_schedule", rc)
    return item_cta.view(B * H, n_tiles), cta_q_tiles


def fattn_bwd_schedule_items(B: int, H: int, N: int, d: int, causal: bool, grid: int,
                             l2_bytes: int, deterministic: bool = False):
    """The backward schedule in processing order (host only): a list, per CTA,
    of its items (bh, j, i0, n_it, rot) in the order it runs them."""
    n_items = B * H * ((N + 127) // 128)
    start = torch.empty(max(grid, 0) + 1, dtype=torch.int32)
    items = torch.empty(5 * n_items, dtype=torch.int32)
    rc = _lib.load().fattn_bwd_schedule_items(B, H, N, d, int(bool(causal)),
                                              int(bool(deterministic)), grid, l2_bytes,
                                              start.data_ptr(), items.data_ptr())
    _lib.check("fattn_bwd_schedule_items", rc)
    it = items.view(n_items, 5).tolist()
    st = start.tolist()
    return [[tuple(e) for e in it[st[c]:st[c + 1]]] for c in range(grid)]


def fattn_bwd_pair_schedule_items(B: int, H: int, N: int, causal: bool, clusters: int,
                                  l2_bytes: int):
    """The CTA-pair backward's schedule (host only): per cluster, its units
    (bh, 2u, i0, n_it, rot) in processing order."""
    n_units = B * H * (((N + 127) // 128 + 1) // 2)
    start = torch.empty(max(clusters, 0) + 1, dtype=torch.int32)
    items = torch.empty(5 * n_units, dtype=torch.int32)
    rc = _lib.load().fattn_bwd_pair_schedule_items(B, H, N, int(bool(causal)), clusters, l2_bytes,
                                                   start.data_ptr(), items.data_ptr())
    _lib.check("fattn_bwd_pair_schedule_items", rc)
    it = items.view(n_units, 5).tolist()
    st = start.tolist()
    return [[tuple(e) for e in it[st[c]:st[c + 1]]] for c in range(clusters)]


def fattn_check_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the status."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    lib = _lib.load()
    with torch.cuda.device(dev):
        return int(lib.fattn_check_status(_stream_ptr(dev)))


def fattn_set_wait_budget(cycles: int) -> None:
    _lib.load().fattn_set_wait_budget(int(cycles))


def fattn_set_rescale_threshold(tau_log2: float) -> None:
    _lib.load().fattn_set_rescale_threshold(float(tau_log2))


def fattn_set_deterministic(on: bool) -> None:
    """dQ accumulated in a fixed order (bitwise reproducible backward)."""
    _lib.load().fattn_set_deterministic(1 if on else 0)


def fattn_set_bwd_pair(on: bool) -> None:
    """d = 128 backward: CTA pairs (True) or one CTA per K/V tile (False, the default)."""
    _lib.load().fattn_set_bwd_pair(int(bool(on)))


def fattn_selftest_timeout(budget_cycles: int, device=None) -> int:
    dev = torch.device("cuda") if device is None else torch.device(device)
    lib = _lib.load()
    with torch.cuda.device(dev):
        return int(lib.fattn_selftest_timeout(int(budget_cycles), _stream_ptr(dev)))
