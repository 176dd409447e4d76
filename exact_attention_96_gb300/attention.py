"""PyTorch-facing calls: device memory and the current stream come from torch; all
arithmetic runs in libfa_gb300.so (include/fa.h).  Tensors are bf16, contiguous,
[B, H, N, d] on a CUDA device; LSE is fp32 [B, H, N].
"""

from __future__ import annotations

import math

import torch

from . import abi


def _check_qkv(*ts):
    t0 = ts[0]
    if t0.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    for t in ts:
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("expected contiguous bf16 CUDA tensors")
        if t.shape != t0.shape or t.device != t0.device:
            raise ValueError("all tensors must share shape and device")


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
            dropout_p: float = 0.0, seed: int = 0):
    """O, LSE = attention(q, k, v); writes into `out` / `lse` when given.  dropout_p > 0
    applies the generator-defined dropout mask of (seed, head, query, key) (fa_fwd_dropout)."""
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    with torch.cuda.device(q.device):
        if dropout_p > 0:
            st = abi.fa_fwd_dropout(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                                    B, H, N, d, scale, causal, dropout_p, seed, _stream(q))
        else:
            st = abi.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                            B, H, N, d, scale, causal, _stream(q))
    abi.check("fa_fwd_dropout" if dropout_p > 0 else "fa_fwd", st)
    return o, l


def forward_fp8(q8, k8, vt8, q_descale: float, k_descale: float, v_descale: float,
                causal: bool = False, scale: float | None = None, out=None, lse=None):
    """FP8 forward, head dim 128: q8, k8 uint8 E4M3 codes [B, H, N, 128]; vt8 the codes of V
    transposed, uint8 [B, H, 128, ldv] with ldv >= N a multiple of 16.  Returns bf16 O and
    fp32 LSE of attention over the real inputs descale * code."""
    for t in (q8, k8, vt8):
        if not t.is_cuda or t.dtype != torch.uint8 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("expected contiguous uint8 CUDA tensors of rank 4")
    B, H, N, d = q8.shape
    if k8.shape != q8.shape or vt8.shape[:3] != (B, H, d):
        raise ValueError("k8 must match q8; vt8 must be [B, H, d, ldv]")
    ldv = vt8.shape[3]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    l = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    with torch.cuda.device(q8.device):
        st = abi.fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), ldv, o.data_ptr(), l.data_ptr(),
                            B, H, N, d, scale, q_descale, k_descale, v_descale, causal, _stream(q8))
    abi.check("fa_fwd_fp8", st)
    return o, l


def quantize_fp8(x, transpose: bool = False, ld: int | None = None, descale=None):
    """E4M3 codes of a bf16 [B, H, N, d] tensor and its fp32 descale (a 1-element CUDA tensor):
    descale = max|x| / 448 (fa_e4m3_descale) unless given, codes = E4M3(x / descale)
    (fa_quantize_e4m3).  transpose=True gives the [B, H, d, ld] layout of V for forward_fp8
    (ld defaults to N rounded up to 16)."""
    _check_qkv(x)
    B, H, N, d = x.shape
    with torch.cuda.device(x.device):
        if descale is None:
            descale = torch.empty(1, dtype=torch.float32, device=x.device)
            abi.check("fa_e4m3_descale", abi.fa_e4m3_descale(x.data_ptr(), x.numel(), descale.data_ptr(),
                                                             _stream(x)))
        if transpose:
            ld = (N + 15) // 16 * 16 if ld is None else int(ld)
            out = torch.empty((B, H, d, ld), dtype=torch.uint8, device=x.device)
        else:
            ld = 0
            out = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device)
        abi.check("fa_quantize_e4m3", abi.fa_quantize_e4m3(x.data_ptr(), out.data_ptr(), B, H, N, d, transpose, ld,
                                                           descale.data_ptr(), _stream(x)))
    return out, descale


def forward_fp8_from_bf16(q, k, v, causal: bool = False, scale: float | None = None):
    """The FP8 forward of bf16 inputs: each of Q, K, V is quantised on the device with its own
    descale (quantize_fp8; V transposed), the three descales are read back (one small
    device-to-host copy) and passed to forward_fp8.  Returns (O, LSE, (q8, k8, vt8),
    (q_descale, k_descale, v_descale))."""
    _check_qkv(q, k, v)
    q8, qs = quantize_fp8(q)
    k8, ks = quantize_fp8(k)
    vt8, vs = quantize_fp8(v, transpose=True)
    qs_h, ks_h, vs_h = torch.cat([qs, ks, vs]).tolist()
    o, l = forward_fp8(q8, k8, vt8, qs_h, ks_h, vs_h, causal=causal, scale=scale)
    return o, l, (q8, k8, vt8), (qs_h, ks_h, vs_h)


def forward_splitkv(q, k, v, num_splits: int = 0, scale: float | None = None, out=None, lse=None,
                    workspace=None):
    """Split-KV forward (no mask): q [B,H,Nq,d] against k, v [B,H,Nk,d]; returns (O, LSE)."""
    for t in (q, k, v):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("expected contiguous bf16 CUDA tensors [B, H, N, d]")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, H, Nk, d] with q's B, H, d")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    nbytes = abi.fa_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        st = abi.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), l.data_ptr(),
                                B, H, Nq, Nk, d, scale, num_splits, workspace.data_ptr(),
                                workspace.numel(), _stream(q))
    abi.check("fa_fwd_splitkv", st)
    return o, l


def workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return abi.fa_bwd_workspace_bytes(B, H, N, d)


def backward(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None,
             workspace=None, grads=None, dropout_p: float = 0.0, seed: int = 0):
    """dQ, dK, dV of attention for upstream gradient `do` (O and LSE from forward; with
    dropout, the forward's dropout_p and seed)."""
    _check_qkv(q, k, v, o, do)
    B, H, N, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    nbytes = workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    dq, dk, dv = grads
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr())
    with torch.cuda.device(q.device):
        if dropout_p > 0:
            st = abi.fa_bwd_dropout(*ptrs, B, H, N, d, scale, causal, dropout_p, seed,
                                    workspace.data_ptr(), workspace.numel(), _stream(q))
        else:
            st = abi.fa_bwd(*ptrs, B, H, N, d, scale, causal, workspace.data_ptr(), workspace.numel(),
                            _stream(q))
    abi.check("fa_bwd_dropout" if dropout_p > 0 else "fa_bwd", st)
    return dq, dk, dv


def step_host(q_h, k_h, v_h, do_h, causal: bool = False, scale: float | None = None, out=None,
              device_buffers=None, workspace=None, num_chunks: int = 0, device=None):
    """One forward + backward step with inputs and results in host memory (fa_step_host):
    the copies of one chunk of heads overlap the kernels of another.  q_h, k_h, v_h, do_h:
    pinned CPU bf16 [B, H, N, d].  Returns the host results (O, LSE, dQ, dK, dV), written into
    `out` when given.  device_buffers (q, k, v, dO, O, LSE, dQ, dK, dV on the device) and
    workspace are allocated when not given; pass them to reuse them across steps.  The call
    is asynchronous on the current stream, like the others."""
    for t in (q_h, k_h, v_h, do_h):
        if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("expected contiguous bf16 host tensors [B, H, N, d]")
    B, H, N, d = q_h.shape
    dev = torch.device("cuda") if device is None else torch.device(device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = tuple(torch.empty(q_h.shape, dtype=torch.bfloat16).pin_memory() for _ in range(4))
        out = (out[0], torch.empty((B, H, N), dtype=torch.float32).pin_memory(), *out[1:])
    if device_buffers is None:
        device_buffers = [torch.empty(q_h.shape, dtype=torch.bfloat16, device=dev) for _ in range(5)]
        device_buffers += [torch.empty((B, H, N), dtype=torch.float32, device=dev)]
        device_buffers += [torch.empty(q_h.shape, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    if workspace is None:
        workspace = torch.empty(abi.fa_step_host_workspace_bytes(B, H, N, d, num_chunks), dtype=torch.uint8,
                                device=dev)
    host_ptrs = [t.data_ptr() for t in (q_h, k_h, v_h, do_h, *out)]
    dev_ptrs = [t.data_ptr() for t in device_buffers]
    with torch.cuda.device(dev):
        st = abi.fa_step_host(host_ptrs, dev_ptrs, B, H, N, d, scale, causal, num_chunks,
                              workspace.data_ptr(), workspace.numel(), torch.cuda.current_stream(dev).cuda_stream)
    abi.check("fa_step_host", st)
    return out


def status_check(device=None) -> int:
    """Synchronises the current stream and returns the library's device status code."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return abi.fa_status_check(torch.cuda.current_stream(dev).cuda_stream)
