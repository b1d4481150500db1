"""DFlash2 draft-block head on one GB300: Python binding of libdflash2.

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are torch CUDA tensors (bf16 weights/activations as torch.bfloat16),
contiguous and row-major; calls are asynchronous on the current torch stream.

    ids, vals, G = unary_topk(h, W_lm, K, W_H)          # logits never leave the chip
    path, scores = selector_walk(anchors, ids, vals, G, A, Bc, block_size)
    s = selector_pair_scores(pred, ids, vals, G, A, Bc)  # teacher-forced
    loss, label = selector_ce(s, ids, targets, V)      # the selector's K-way CE
    y, dyn = conv_prepare(x, block_size, taps, group, W_proj, base)
    y2 = conv_finish(z, block_size, taps, group, dyn, base)
"""
from __future__ import annotations

import ctypes as ct

import torch

from . import _abi

DF2_DTYPE_BF16 = 0
DF2_DTYPE_F32 = 1
DF2_STATUS_ID_OUT_OF_RANGE = 0x1
DF2_STATUS_WAIT_TIMEOUT = 0x2
DF2_HEAD_PATH_STREAM = 0
DF2_HEAD_PATH_GEMM = 1
DF2_HEAD_PATH_CUDA_CORE = 2


class DFlash2Error(RuntimeError):
    def __init__(self, call: str, code: int):
        self.code = code
        super().__init__(f"{call}: {status_string(code)}")


def lib():
    return _abi.load()


def kernels_launched() -> int:
    """Kernels this library has launched in this process so far."""
    return int(lib().dflash2_kernels_launched())


def unary_topk_path(P, D, V, K) -> int:
    """DF2_HEAD_PATH_* of the head kernels for these shapes (-1: shapes rejected)."""
    return int(lib().dflash2_unary_topk_path(P, D, V, K))


def status_string(code: int) -> str:
    return lib().dflash2_status_string(int(code)).decode()


def _p(t):
    return ct.c_void_p(t.data_ptr() if t is not None else 0)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ct.c_void_p(s.cuda_stream)


def _need(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def _check(call, rc):
    if rc != 0:
        raise DFlash2Error(call, rc)


def _workspace(nbytes, workspace, device):
    if nbytes == 0:
        return None
    if workspace is None:
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace too small: need {nbytes} bytes")
    return workspace


def unary_topk_workspace_size(P, D, V, K, r=0) -> int:
    return int(lib().dflash2_unary_topk_workspace_size(P, D, V, K, r))


def unary_topk(h, W_lm, K, W_H=None, *, output_multiplier=1.0, final_logit_softcapping=0.0,
               workspace=None, dev_status=None, out=None, stream=None):
    """Top-K unary logits per row of h, and G = h W_H^T.  Returns (ids, vals, G).

    output_multiplier m and final_logit_softcapping c map each logit u to
    c*tanh(m*u/c) (m*u when c = 0) before the selection; the defaults leave it."""
    _need(h, "h", torch.bfloat16, 2)
    _need(W_lm, "W_lm", torch.bfloat16, 2)
    P, D = h.shape
    V = W_lm.shape[0]
    if W_lm.shape[1] != D:
        raise ValueError("W_lm must be [V, D]")
    r = 0
    if W_H is not None:
        _need(W_H, "W_H", torch.bfloat16, 2)
        r = W_H.shape[0]
        if W_H.shape[1] != D:
            raise ValueError("W_H must be [r, D]")
    dev = h.device
    if out is None:
        ids = torch.empty((P, K), dtype=torch.int32, device=dev)
        vals = torch.empty((P, K), dtype=torch.float32, device=dev)
        G = torch.empty((P, r), dtype=torch.float32, device=dev) if r else None
    else:
        ids, vals, G = out
    ws = _workspace(unary_topk_workspace_size(P, D, V, K, r), workspace, dev)
    rc = lib().dflash2_unary_topk(_p(h), P, D, _p(W_lm), V, int(K), float(output_multiplier),
                                  float(final_logit_softcapping), _p(W_H), r, _p(G), _p(ids),
                                  _p(vals), _p(ws), 0 if ws is None else ws.numel(),
                                  _p(dev_status), _stream(stream))
    _check("dflash2_unary_topk", rc)
    return ids, vals, G


def unary_topk_noalloc(h, W_lm, K, W_H=None, *, output_multiplier=1.0, final_logit_softcapping=0.0,
                       dev_status=None, out=None, stream=None):
    """unary_topk without a workspace: for callers that may not allocate device
    memory during a call.  Scratch comes from a fixed array inside the library
    (DF2_NOALLOC_SCRATCH_BYTES per GPU), shared by every call, so calls must not
    overlap on the GPU.  Outputs are allocated here unless `out` is given."""
    _need(h, "h", torch.bfloat16, 2)
    _need(W_lm, "W_lm", torch.bfloat16, 2)
    P, D = h.shape
    r = 0 if W_H is None else W_H.shape[0]
    if out is None:
        ids = torch.empty((P, K), dtype=torch.int32, device=h.device)
        vals = torch.empty((P, K), dtype=torch.float32, device=h.device)
        G = torch.empty((P, r), dtype=torch.float32, device=h.device) if r else None
    else:
        ids, vals, G = out
    rc = lib().dflash2_unary_topk_noalloc(_p(h), P, D, _p(W_lm), W_lm.shape[0], int(K),
                                          float(output_multiplier), float(final_logit_softcapping), _p(W_H), r,
                                          _p(G), _p(ids), _p(vals), _p(dev_status), _stream(stream))
    _check("dflash2_unary_topk_noalloc", rc)
    return ids, vals, G


def selector_walk(anchors, topk_ids, topk_vals, G, A, Bc, block_size, *, dev_status=None,
                  out=None, stream=None):
    """Greedy walk per request.  Returns (path [R, B-1] int32, path_scores [R, B-1] f32)."""
    _need(anchors, "anchors", torch.int32, 1)
    _need(topk_ids, "topk_ids", torch.int32)
    _need(topk_vals, "topk_vals", torch.float32)
    _need(G, "G", torch.float32)
    _need(A, "A", torch.bfloat16, 2)
    _need(Bc, "Bc", torch.bfloat16, 2)
    R = anchors.shape[0]
    B = int(block_size)
    K = topk_ids.shape[-1]
    V, r = A.shape
    if topk_ids.numel() != R * B * K or topk_vals.numel() != R * B * K or G.numel() != R * B * r:
        raise ValueError("candidate / gate shapes do not match [R*B, K] / [R*B, r]")
    if tuple(Bc.shape) != (V, r):
        raise ValueError("Bc must be [V, r] like A")
    if out is None:
        path = torch.empty((R, B - 1), dtype=torch.int32, device=anchors.device)
        scores = torch.empty((R, B - 1), dtype=torch.float32, device=anchors.device)
    else:
        path, scores = out
    rc = lib().dflash2_selector_walk(_p(anchors), R, B, _p(topk_ids), _p(topk_vals), _p(G), _p(A),
                                     _p(Bc), V, K, r, _p(path), _p(scores), _p(dev_status),
                                     _stream(stream))
    _check("dflash2_selector_walk", rc)
    return path, scores


def selector_ce(scores, topk_ids, targets, V, *, dev_status=None, out=None, stream=None):
    """The selector's K-way cross-entropy per row of teacher-forced scores [P, K]:
    (loss [P] fp32, label [P] int32); rows whose target is not a candidate give
    label -1 and NaN loss."""
    _need(scores, "scores", torch.float32)
    _need(topk_ids, "topk_ids", torch.int32)
    _need(targets, "targets", torch.int32, 1)
    P = targets.shape[0]
    K = topk_ids.shape[-1]
    if topk_ids.numel() != P * K or scores.numel() != P * K:
        raise ValueError("scores / topk_ids do not match [P, K]")
    if out is None:
        out = (torch.empty((P,), dtype=torch.float32, device=scores.device),
               torch.empty((P,), dtype=torch.int32, device=scores.device))
    loss, label = out
    rc = lib().dflash2_selector_ce(_p(scores), _p(topk_ids), _p(targets), P, K, int(V), _p(loss), _p(label),
                                   _p(dev_status), _stream(stream))
    _check("dflash2_selector_ce", rc)
    return loss, label


def selector_pair_scores(pred, topk_ids, topk_vals, G, A, Bc, *, dev_status=None, out=None,
                         stream=None):
    """Teacher-forced scores [P, K]."""
    _need(pred, "pred", torch.int32, 1)
    _need(topk_ids, "topk_ids", torch.int32)
    _need(topk_vals, "topk_vals", torch.float32)
    _need(G, "G", torch.float32)
    _need(A, "A", torch.bfloat16, 2)
    _need(Bc, "Bc", torch.bfloat16, 2)
    P = pred.shape[0]
    K = topk_ids.shape[-1]
    V, r = A.shape
    if topk_ids.numel() != P * K or topk_vals.numel() != P * K or G.numel() != P * r:
        raise ValueError("candidate / gate shapes do not match [P, K] / [P, r]")
    scores = out if out is not None else torch.empty((P, K), dtype=torch.float32, device=pred.device)
    rc = lib().dflash2_selector_pair_scores(_p(pred), P, _p(topk_ids), _p(topk_vals), _p(G), _p(A),
                                            _p(Bc), V, K, r, _p(scores), _p(dev_status),
                                            _stream(stream))
    _check("dflash2_selector_pair_scores", rc)
    return scores


def draft_head_workspace_size(R, B, D, V, K, r) -> int:
    return int(lib().dflash2_draft_head_workspace_size(R, B, D, V, K, r))


def draft_head(h, W_lm, K, W_H, A, Bc, anchors, block_size, pred=None, *, output_multiplier=1.0,
               final_logit_softcapping=0.0, workspace=None, dev_status=None, out=None, stream=None):
    """Unary top-K, G = H(h), the greedy walk and (pred given) the teacher-forced
    scores of one draft block in one call.  Returns (ids, vals, G, path, path_scores,
    pair_scores or None)."""
    _need(h, "h", torch.bfloat16, 2)
    _need(W_lm, "W_lm", torch.bfloat16, 2)
    _need(W_H, "W_H", torch.bfloat16, 2)
    _need(A, "A", torch.bfloat16, 2)
    _need(Bc, "Bc", torch.bfloat16, 2)
    _need(anchors, "anchors", torch.int32, 1)
    P, D = h.shape
    V = W_lm.shape[0]
    r = W_H.shape[0]
    R = anchors.shape[0]
    B = int(block_size)
    if P != R * B or W_lm.shape[1] != D or W_H.shape[1] != D:
        raise ValueError("h must be [R*B, D] with W_lm [V, D], W_H [r, D]")
    if tuple(A.shape) != (V, r) or tuple(Bc.shape) != (V, r):
        raise ValueError("A and Bc must be [V, r]")
    if pred is not None:
        _need(pred, "pred", torch.int32, 1)
        if pred.shape[0] != P:
            raise ValueError("pred must be [R*B]")
    dev = h.device
    if out is None:
        e = torch.empty
        out = (e((P, K), dtype=torch.int32, device=dev), e((P, K), dtype=torch.float32, device=dev),
               e((P, r), dtype=torch.float32, device=dev), e((R, B - 1), dtype=torch.int32, device=dev),
               e((R, B - 1), dtype=torch.float32, device=dev),
               e((P, K), dtype=torch.float32, device=dev) if pred is not None else None)
    ids, vals, G, path, ps, pair = out
    need = draft_head_workspace_size(R, B, D, V, K, r)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    rc = lib().dflash2_draft_head(_p(h), R, B, D, _p(W_lm), V, K, float(output_multiplier),
                                  float(final_logit_softcapping), _p(W_H), r, _p(A), _p(Bc), _p(anchors),
                                  _p(pred), _p(ids), _p(vals), _p(G), _p(path), _p(ps), _p(pair),
                                  _p(workspace), workspace.numel(), _p(dev_status), _stream(stream))
    _check("dflash2_draft_head", rc)
    return ids, vals, G, path, ps, pair


def selector_lattice(anchors, topk_ids, topk_vals, G, A, Bc, block_size, *, dev_status=None,
                     out=None, stream=None):
    """Every adjacent candidate pair scored at once: lattice [R, B-1, K, K] f32."""
    _need(anchors, "anchors", torch.int32, 1)
    _need(topk_ids, "topk_ids", torch.int32)
    _need(topk_vals, "topk_vals", torch.float32)
    _need(G, "G", torch.float32)
    _need(A, "A", torch.bfloat16, 2)
    _need(Bc, "Bc", torch.bfloat16, 2)
    R = anchors.shape[0]
    B = int(block_size)
    K = topk_ids.shape[-1]
    V, r = A.shape
    if topk_ids.numel() != R * B * K or topk_vals.numel() != R * B * K or G.numel() != R * B * r:
        raise ValueError("candidate / gate shapes do not match [R*B, K] / [R*B, r]")
    if tuple(Bc.shape) != (V, r):
        raise ValueError("Bc must be [V, r] like A")
    lat = out if out is not None else torch.empty((R, B - 1, K, K), dtype=torch.float32,
                                                  device=anchors.device)
    _need(lat, "lattice", torch.float32)
    if lat.numel() != R * (B - 1) * K * K:
        raise ValueError("lattice must hold [R, B-1, K, K]")
    rc = lib().dflash2_selector_lattice(_p(anchors), R, B, _p(topk_ids), _p(topk_vals), _p(G), _p(A),
                                        _p(Bc), V, K, r, _p(lat), _p(dev_status), _stream(stream))
    _check("dflash2_selector_lattice", rc)
    return lat


def lattice_walk(lattice, topk_ids, block_size, vocab_size, *, uniforms=None, temperature=1.0,
                 dev_status=None, out=None, stream=None):
    """Greedy (uniforms None) or sampling walk over a lattice.  Returns (path [R, B-1]
    int32, path_scores [R, B-1] f32)."""
    _need(lattice, "lattice", torch.float32, 4)
    _need(topk_ids, "topk_ids", torch.int32)
    R, T, K, K2 = lattice.shape
    B = int(block_size)
    if K2 != K or T != B - 1 or topk_ids.numel() != R * B * K:
        raise ValueError("lattice must be [R, B-1, K, K] over topk_ids [R*B, K]")
    if uniforms is not None:
        _need(uniforms, "uniforms", torch.float32)
        if uniforms.numel() != R * T:
            raise ValueError("uniforms must be [R, B-1]")
    if out is None:
        path = torch.empty((R, T), dtype=torch.int32, device=lattice.device)
        scores = torch.empty((R, T), dtype=torch.float32, device=lattice.device)
    else:
        path, scores = out
    rc = lib().dflash2_lattice_walk(_p(lattice), _p(topk_ids), R, B, K, int(vocab_size), _p(uniforms),
                                    float(temperature), _p(path), _p(scores), _p(dev_status),
                                    _stream(stream))
    _check("dflash2_lattice_walk", rc)
    return path, scores


def _act_dtype(x):
    if x.dtype == torch.bfloat16:
        return DF2_DTYPE_BF16
    if x.dtype == torch.float32:
        return DF2_DTYPE_F32
    raise TypeError("conv activations must be bfloat16 or float32")


def conv_prepare_workspace_size(P, C, taps, group, dtype=DF2_DTYPE_BF16) -> int:
    return int(lib().dflash2_conv_prepare_workspace_size(P, C, taps, group, dtype))


def conv_prepare(x, block_size, taps, group, W_proj, base, *, workspace=None, out=None, stream=None):
    """Conv before a sublayer.  Returns (y like x, dyn_out [P, taps, C/group] f32)."""
    dt = _act_dtype(x)
    _need(x, "x", x.dtype, 2)
    _need(W_proj, "W_proj", torch.bfloat16, 2)
    _need(base, "base", torch.float32, 3)
    P, C = x.shape
    G = C // group
    if out is None:
        y = torch.empty_like(x)
        dyn = torch.empty((P, taps, G), dtype=torch.float32, device=x.device)
    else:
        y, dyn = out
    ws = _workspace(conv_prepare_workspace_size(P, C, taps, group, dt), workspace, x.device)
    rc = lib().dflash2_conv_prepare(_p(x), dt, P, C, int(block_size), int(taps), int(group),
                                    _p(W_proj), _p(base), _p(y), _p(dyn), _p(ws),
                                    0 if ws is None else ws.numel(), _stream(stream))
    _check("dflash2_conv_prepare", rc)
    return y, dyn


def conv_finish(z, block_size, taps, group, dyn_out, base, *, out=None, stream=None):
    """Conv after the sublayer with prepare's dynamic kernel.  Returns y like z."""
    dt = _act_dtype(z)
    _need(z, "z", z.dtype, 2)
    _need(dyn_out, "dyn_out", torch.float32, 3)
    _need(base, "base", torch.float32, 3)
    P, C = z.shape
    y = out if out is not None else torch.empty_like(z)
    rc = lib().dflash2_conv_finish(_p(z), dt, P, C, int(block_size), int(taps), int(group),
                                   _p(dyn_out), _p(base), _p(y), _stream(stream))
    _check("dflash2_conv_finish", rc)
    return y


def conv_finish_prepare(z, block_size, taps, group, dyn_out, base, W_proj, base_next, residual=None, *,
                        workspace=None, out=None, stream=None):
    """A sublayer's conv finish, plus the residual stream when given, then the next
    sublayer's conv prepare.  Returns (h like z, y_next like z, dyn_out_next
    [P, taps, C/group] f32)."""
    dt = _act_dtype(z)
    _need(z, "z", z.dtype, 2)
    _need(dyn_out, "dyn_out", torch.float32, 3)
    _need(base, "base", torch.float32, 3)
    _need(W_proj, "W_proj", torch.bfloat16, 2)
    _need(base_next, "base_next", torch.float32, 3)
    if residual is not None:
        _need(residual, "residual", z.dtype, 2)
        if residual.shape != z.shape:
            raise ValueError("residual must have z's shape")
    P, C = z.shape
    G = C // group
    if out is None:
        h, y = torch.empty_like(z), torch.empty_like(z)
        dyn = torch.empty((P, taps, G), dtype=torch.float32, device=z.device)
    else:
        h, y, dyn = out
    ws = _workspace(int(lib().dflash2_conv_finish_prepare_workspace_size(P, C, taps, group, dt)), workspace,
                    z.device)
    rc = lib().dflash2_conv_finish_prepare(_p(z), dt, P, C, int(block_size), int(taps), int(group), _p(dyn_out),
                                           _p(base), _p(residual), _p(h), _p(W_proj), _p(base_next), _p(y),
                                           _p(dyn), _p(ws), 0 if ws is None else ws.numel(), _stream(stream))
    _check("dflash2_conv_finish_prepare", rc)
    return h, y, dyn
