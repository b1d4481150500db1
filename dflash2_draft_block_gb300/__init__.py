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


def _on_device(t):
    return t.is_cuda


def _stream(stream, device):
    """The CUDA stream handle of `stream` (default: the current one), which must
    belong to the device of the call's tensors."""
    s = stream if stream is not None else torch.cuda.current_stream()
    if s.device != device:
        raise ValueError(f"the stream is on {s.device}, the call's tensors on {device}")
    return ct.c_void_p(s.cuda_stream)


def _need(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor) or not _on_device(t):
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def _device(first, **others):
    """The device of the call: `first`'s, which every other given tensor shares and
    which is the current CUDA device (the library launches on the current device)."""
    dev = first.device
    for name, t in others.items():
        if t is not None and t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the call's tensors on {dev}")
    if dev.type == "cuda" and dev.index is not None and dev.index != torch.cuda.current_device():
        raise ValueError(f"the tensors are on {dev} but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()} (torch.cuda.set_device first)")
    return dev


def _out(t, name, dtype, numel, dev):
    """A caller-given output: a contiguous tensor of the call's device, dtype and
    element count (the kernels write numel elements through its pointer)."""
    _need(t, name, dtype)
    if t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} elements, got shape {tuple(t.shape)}")
    if t.device != dev:
        raise ValueError(f"{name} is on {t.device}, the call's tensors on {dev}")
    return t


def _status(st, dev):
    """dev_status: None, or one int32 word (at least) on the call's device."""
    if st is not None:
        _need(st, "dev_status", torch.int32)
        if st.numel() < 1 or st.device != dev:
            raise ValueError("dev_status must hold an int32 word on the call's device")
    return st


def _check(call, rc):
    if rc != 0:
        raise DFlash2Error(call, rc)


def _workspace(nbytes, workspace, device):
    if nbytes == 0 and workspace is None:
        return None
    if workspace is None:
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    _need(workspace, "workspace", workspace.dtype)
    if workspace.device != device:
        raise ValueError(f"workspace is on {workspace.device}, the call's tensors on {device}")
    if _nbytes(workspace) < nbytes:
        raise ValueError(f"workspace too small: need {nbytes} bytes")
    return workspace


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


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
    dev = _device(h, W_lm=W_lm, W_H=W_H)
    if out is None:
        ids = torch.empty((P, K), dtype=torch.int32, device=dev)
        vals = torch.empty((P, K), dtype=torch.float32, device=dev)
        G = torch.empty((P, r), dtype=torch.float32, device=dev) if r else None
    else:
        ids, vals, G = out
        _out(ids, "ids", torch.int32, P * K, dev)
        _out(vals, "vals", torch.float32, P * K, dev)
        if r:
            _out(G, "G", torch.float32, P * r, dev)
    _status(dev_status, dev)
    ws = _workspace(unary_topk_workspace_size(P, D, V, K, r), workspace, dev)
    rc = lib().dflash2_unary_topk(_p(h), P, D, _p(W_lm), V, int(K), float(output_multiplier),
                                  float(final_logit_softcapping), _p(W_H), r, _p(G), _p(ids),
                                  _p(vals), _p(ws), _nbytes(ws),
                                  _p(dev_status), _stream(stream, dev))
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
    if W_lm.shape[1] != D:
        raise ValueError("W_lm must be [V, D]")
    r = 0
    if W_H is not None:
        _need(W_H, "W_H", torch.bfloat16, 2)
        r = W_H.shape[0]
        if W_H.shape[1] != D:
            raise ValueError("W_H must be [r, D]")
    dev = _device(h, W_lm=W_lm, W_H=W_H)
    if out is None:
        ids = torch.empty((P, K), dtype=torch.int32, device=dev)
        vals = torch.empty((P, K), dtype=torch.float32, device=dev)
        G = torch.empty((P, r), dtype=torch.float32, device=dev) if r else None
    else:
        ids, vals, G = out
        _out(ids, "ids", torch.int32, P * K, dev)
        _out(vals, "vals", torch.float32, P * K, dev)
        if r:
            _out(G, "G", torch.float32, P * r, dev)
    _status(dev_status, dev)
    rc = lib().dflash2_unary_topk_noalloc(_p(h), P, D, _p(W_lm), W_lm.shape[0], int(K),
                                          float(output_multiplier), float(final_logit_softcapping), _p(W_H), r,
                                          _p(G), _p(ids), _p(vals), _p(dev_status), _stream(stream, dev))
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
    dev = _device(anchors, topk_ids=topk_ids, topk_vals=topk_vals, G=G, A=A, Bc=Bc)
    T = max(B - 1, 0)
    if out is None:
        path = torch.empty((R, T), dtype=torch.int32, device=dev)
        scores = torch.empty((R, T), dtype=torch.float32, device=dev)
    else:
        path, scores = out
        _out(path, "path", torch.int32, R * T, dev)
        _out(scores, "path_scores", torch.float32, R * T, dev)
    _status(dev_status, dev)
    rc = lib().dflash2_selector_walk(_p(anchors), R, B, _p(topk_ids), _p(topk_vals), _p(G), _p(A),
                                     _p(Bc), V, K, r, _p(path), _p(scores), _p(dev_status),
                                     _stream(stream, dev))
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
    dev = _device(scores, topk_ids=topk_ids, targets=targets)
    if out is None:
        out = (torch.empty((P,), dtype=torch.float32, device=dev),
               torch.empty((P,), dtype=torch.int32, device=dev))
    loss, label = out
    _out(loss, "loss", torch.float32, P, dev)
    _out(label, "label", torch.int32, P, dev)
    _status(dev_status, dev)
    rc = lib().dflash2_selector_ce(_p(scores), _p(topk_ids), _p(targets), P, K, int(V), _p(loss), _p(label),
                                   _p(dev_status), _stream(stream, dev))
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
    if tuple(Bc.shape) != (V, r):
        raise ValueError("Bc must be [V, r] like A")
    dev = _device(pred, topk_ids=topk_ids, topk_vals=topk_vals, G=G, A=A, Bc=Bc)
    if out is None:
        scores = torch.empty((P, K), dtype=torch.float32, device=dev)
    else:
        scores = _out(out, "scores", torch.float32, P * K, dev)
    _status(dev_status, dev)
    rc = lib().dflash2_selector_pair_scores(_p(pred), P, _p(topk_ids), _p(topk_vals), _p(G), _p(A),
                                            _p(Bc), V, K, r, _p(scores), _p(dev_status),
                                            _stream(stream, dev))
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
    dev = _device(h, W_lm=W_lm, W_H=W_H, A=A, Bc=Bc, anchors=anchors, pred=pred)
    T = max(B - 1, 0)
    if out is None:
        e = torch.empty
        out = (e((P, K), dtype=torch.int32, device=dev), e((P, K), dtype=torch.float32, device=dev),
               e((P, r), dtype=torch.float32, device=dev), e((R, T), dtype=torch.int32, device=dev),
               e((R, T), dtype=torch.float32, device=dev),
               e((P, K), dtype=torch.float32, device=dev) if pred is not None else None)
    ids, vals, G, path, ps, pair = out
    _out(ids, "ids", torch.int32, P * K, dev)
    _out(vals, "vals", torch.float32, P * K, dev)
    _out(G, "G", torch.float32, P * r, dev)
    _out(path, "path", torch.int32, R * T, dev)
    _out(ps, "path_scores", torch.float32, R * T, dev)
    if pred is not None:
        _out(pair, "pair_scores", torch.float32, P * K, dev)
    _status(dev_status, dev)
    workspace = _workspace(draft_head_workspace_size(R, B, D, V, K, r), workspace, dev)
    if workspace is None:  # nothing to hold (R = 0): the call still takes a buffer
        workspace = torch.empty(1, dtype=torch.uint8, device=dev)
    rc = lib().dflash2_draft_head(_p(h), R, B, D, _p(W_lm), V, K, float(output_multiplier),
                                  float(final_logit_softcapping), _p(W_H), r, _p(A), _p(Bc), _p(anchors),
                                  _p(pred), _p(ids), _p(vals), _p(G), _p(path), _p(ps), _p(pair),
                                  _p(workspace), _nbytes(workspace), _p(dev_status), _stream(stream, dev))
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
    dev = _device(anchors, topk_ids=topk_ids, topk_vals=topk_vals, G=G, A=A, Bc=Bc)
    T = max(B - 1, 0)
    lat = out if out is not None else torch.empty((R, T, K, K), dtype=torch.float32, device=dev)
    _out(lat, "lattice", torch.float32, R * T * K * K, dev)
    _status(dev_status, dev)
    rc = lib().dflash2_selector_lattice(_p(anchors), R, B, _p(topk_ids), _p(topk_vals), _p(G), _p(A),
                                        _p(Bc), V, K, r, _p(lat), _p(dev_status), _stream(stream, dev))
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
    dev = _device(lattice, topk_ids=topk_ids, uniforms=uniforms)
    if out is None:
        path = torch.empty((R, T), dtype=torch.int32, device=dev)
        scores = torch.empty((R, T), dtype=torch.float32, device=dev)
    else:
        path, scores = out
        _out(path, "path", torch.int32, R * T, dev)
        _out(scores, "path_scores", torch.float32, R * T, dev)
    _status(dev_status, dev)
    rc = lib().dflash2_lattice_walk(_p(lattice), _p(topk_ids), R, B, K, int(vocab_size), _p(uniforms),
                                    float(temperature), _p(path), _p(scores), _p(dev_status),
                                    _stream(stream, dev))
    _check("dflash2_lattice_walk", rc)
    return path, scores


def _act_dtype(x):
    if x.dtype == torch.bfloat16:
        return DF2_DTYPE_BF16
    if x.dtype == torch.float32:
        return DF2_DTYPE_F32
    raise TypeError("conv activations must be bfloat16 or float32")


def _conv_shapes(C, taps, group, **named):
    """The conv's weight and correction shapes (skipped when taps or group are
    themselves invalid: the library rejects those with a status)."""
    if not (taps >= 1 and group >= 1 and C % group == 0):
        return
    G = C // group
    want = {"W_proj": (2 * taps * G, C), "base": (2, taps, C), "base_next": (2, taps, C)}
    for name, (t, P) in named.items():
        shape = (P, taps, G) if name == "dyn_out" else want[name]
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must be {list(shape)}, got {list(t.shape)}")


def conv_prepare_workspace_size(P, C, taps, group, dtype=DF2_DTYPE_BF16) -> int:
    return int(lib().dflash2_conv_prepare_workspace_size(P, C, taps, group, dtype))


def conv_prepare(x, block_size, taps, group, W_proj, base, *, workspace=None, out=None, stream=None):
    """Conv before a sublayer.  Returns (y like x, dyn_out [P, taps, C/group] f32)."""
    dt = _act_dtype(x)
    _need(x, "x", x.dtype, 2)
    _need(W_proj, "W_proj", torch.bfloat16, 2)
    _need(base, "base", torch.float32, 3)
    P, C = x.shape
    taps, group = int(taps), int(group)
    _conv_shapes(C, taps, group, W_proj=(W_proj, P), base=(base, P))
    G = C // group if group >= 1 else 0
    dev = _device(x, W_proj=W_proj, base=base)
    if out is None:
        y = torch.empty_like(x)
        dyn = torch.empty((P, taps, G), dtype=torch.float32, device=dev)
    else:
        y, dyn = out
        _out(y, "y", x.dtype, P * C, dev)
        _out(dyn, "dyn_out", torch.float32, P * max(taps, 0) * G, dev)
    ws = _workspace(conv_prepare_workspace_size(P, C, taps, group, dt), workspace, dev)
    rc = lib().dflash2_conv_prepare(_p(x), dt, P, C, int(block_size), taps, group,
                                    _p(W_proj), _p(base), _p(y), _p(dyn), _p(ws),
                                    _nbytes(ws), _stream(stream, dev))
    _check("dflash2_conv_prepare", rc)
    return y, dyn


def conv_finish(z, block_size, taps, group, dyn_out, base, *, out=None, stream=None):
    """Conv after the sublayer with prepare's dynamic kernel.  Returns y like z."""
    dt = _act_dtype(z)
    _need(z, "z", z.dtype, 2)
    _need(dyn_out, "dyn_out", torch.float32, 3)
    _need(base, "base", torch.float32, 3)
    P, C = z.shape
    taps, group = int(taps), int(group)
    _conv_shapes(C, taps, group, dyn_out=(dyn_out, P), base=(base, P))
    dev = _device(z, dyn_out=dyn_out, base=base)
    y = _out(out, "y", z.dtype, P * C, dev) if out is not None else torch.empty_like(z)
    rc = lib().dflash2_conv_finish(_p(z), dt, P, C, int(block_size), taps, group,
                                   _p(dyn_out), _p(base), _p(y), _stream(stream, dev))
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
    taps, group = int(taps), int(group)
    _conv_shapes(C, taps, group, dyn_out=(dyn_out, P), base=(base, P), W_proj=(W_proj, P),
                 base_next=(base_next, P))
    G = C // group if group >= 1 else 0
    dev = _device(z, dyn_out=dyn_out, base=base, W_proj=W_proj, base_next=base_next, residual=residual)
    if out is None:
        h, y = torch.empty_like(z), torch.empty_like(z)
        dyn = torch.empty((P, taps, G), dtype=torch.float32, device=dev)
    else:
        h, y, dyn = out
        _out(h, "h", z.dtype, P * C, dev)
        _out(y, "y_next", z.dtype, P * C, dev)
        _out(dyn, "dyn_out_next", torch.float32, P * max(taps, 0) * G, dev)
    ws = _workspace(int(lib().dflash2_conv_finish_prepare_workspace_size(P, C, taps, group, dt)), workspace, dev)
    rc = lib().dflash2_conv_finish_prepare(_p(z), dt, P, C, int(block_size), taps, group, _p(dyn_out),
                                           _p(base), _p(residual), _p(h), _p(W_proj), _p(base_next), _p(y),
                                           _p(dyn), _p(ws), _nbytes(ws), _stream(stream, dev))
    _check("dflash2_conv_finish_prepare", rc)
    return h, y, dyn
