"""CPU oracle for the DFlash2 draft-block head.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s cpu_baseline / reference legs may import this package.  The
product path (``dflash2_draft_block_gb300``) never imports it and shares no
code with it.

The arithmetic lives in ``dflash2_oracle.c`` (plain loops, fp64 accumulation,
full-sort top-K); this module compiles it with gcc and marshals numpy arrays.
bf16 tensors travel as ``uint16`` arrays of raw bfloat16 bit patterns.

Parity status of each function (what pins it is in ``tests/test_oracle_pins.py``):
every public function here is pinned by closed forms, invariants the pages state,
hand-worked golden cases or brute force; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes as ct
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "dflash2_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
# one build per host architecture (x86 and aarch64 hosts share this tree)
DEFAULT_LIB = os.path.join(BUILD_DIR, f"libdflash2_oracle.{platform.machine()}.so")

# Flags: no fast-math and no FMA contraction, so x86 and Arm hosts produce the
# same doubles from the same loops.
CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]

_lock = threading.Lock()
_default = None


def build(source: str = SOURCE, out: str = DEFAULT_LIB, force: bool = False, extra=()) -> str:
    """Compile the oracle C source into a shared library; returns its path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(source):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, *extra, source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def _p(a):
    return ct.c_void_p(a.ctypes.data) if a is not None else ct.c_void_p(0)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


class Oracle:
    """ctypes binding to one build of the oracle library."""

    def __init__(self, path: str):
        self.path = path
        self.lib = ct.CDLL(path)
        L = self.lib
        i64, i32, vp = ct.c_int64, ct.c_int32, ct.c_void_p
        L.df2o_num_threads.restype = ct.c_int
        L.df2o_set_num_threads.argtypes = [ct.c_int]
        L.df2o_set_num_threads.restype = None
        L.df2o_logits.argtypes = [vp, i64, i64, vp, i64, vp]
        L.df2o_unary_topk.argtypes = [vp, i64, i64, vp, i64, i32, ct.c_double, ct.c_double, vp, i32, vp, vp,
                                      vp, vp]
        L.df2o_selector_walk.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, i64, i32, i32, vp, vp, vp, vp]
        L.df2o_selector_pair_scores.argtypes = [vp, i64, vp, vp, vp, vp, vp, i64, i32, i32, vp, vp]
        L.df2o_selector_lattice.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, i64, i32, i32, vp, vp]
        L.df2o_selector_ce.argtypes = [vp, vp, vp, i64, i32, i64, vp, vp, vp]
        L.df2o_lattice_walk.argtypes = [vp, vp, i32, i32, i32, i64, vp, ct.c_double, vp, vp, vp, vp]
        L.df2o_conv_prepare.argtypes = [vp, ct.c_int, i64, i32, i32, i32, i32, vp, vp, vp, vp]
        L.df2o_conv_finish.argtypes = [vp, ct.c_int, i64, i32, i32, i32, i32, vp, vp, vp]
        L.df2o_conv_finish_prepare.argtypes = [vp, ct.c_int, i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                               vp, vp]
        for f in ("df2o_logits", "df2o_unary_topk", "df2o_selector_walk",
                  "df2o_selector_pair_scores", "df2o_conv_prepare", "df2o_conv_finish",
                  "df2o_conv_finish_prepare", "df2o_selector_ce"):
            getattr(L, f).restype = ct.c_int

    def num_threads(self) -> int:
        return int(self.lib.df2o_num_threads())

    def set_num_threads(self, n: int) -> None:
        """Host threads of the following calls (their results do not depend on it)."""
        self.lib.df2o_set_num_threads(int(n))

    @staticmethod
    def _check(rc):
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (code {rc})")

    # -- unary logits / top-K ------------------------------------------------
    def logits(self, h, W):
        h, W = _c(h, np.uint16), _c(W, np.uint16)
        P, D = h.shape
        V = W.shape[0]
        assert W.shape[1] == D
        U = np.empty((P, V), np.float32)
        self._check(self.lib.df2o_logits(_p(h), P, D, _p(W), V, _p(U)))
        return U

    def unary_topk(self, h, W_lm, K, W_H=None, output_multiplier=1.0, final_logit_softcapping=0.0):
        """Returns (ids [P,K] int32, vals [P,K] f32, margin [P] f64, G [P,r] f32 or None).

        output_multiplier m and final_logit_softcapping c map every logit u to c*tanh(m*u/c)
        (m*u when c is 0).  Both are rounded to fp32 first, the
        precision the library takes them in."""
        h, W_lm = _c(h, np.uint16), _c(W_lm, np.uint16)
        P, D = h.shape
        V = W_lm.shape[0]
        assert W_lm.shape[1] == D
        ids = np.empty((P, K), np.int32)
        vals = np.empty((P, K), np.float32)
        margin = np.empty((P,), np.float64)
        G, r = None, 0
        if W_H is not None:
            W_H = _c(W_H, np.uint16)
            r = W_H.shape[0]
            assert W_H.shape[1] == D
            G = np.empty((P, r), np.float32)
        mul, cap = float(np.float32(output_multiplier)), float(np.float32(final_logit_softcapping))
        self._check(self.lib.df2o_unary_topk(_p(h), P, D, _p(W_lm), V, int(K), mul, cap, _p(W_H), r, _p(G),
                                             _p(ids), _p(vals), _p(margin)))
        return ids, vals, margin, G

    # -- selector -------------------------------------------------------------
    def selector_walk(self, anchors, ids, vals, G, A, Bc, block_size):
        """ids/vals [R*B, K], G [R*B, r]; returns (path [R,B-1], score [R,B-1], margin [R,B-1], status)."""
        anchors = _c(anchors, np.int32)
        ids, vals, G = _c(ids, np.int32), _c(vals, np.float32), _c(G, np.float32)
        A, Bc = _c(A, np.uint16), _c(Bc, np.uint16)
        R = anchors.shape[0]
        B = int(block_size)
        K = ids.shape[-1]
        V, r = A.shape
        assert ids.size == R * B * K and G.size == R * B * r and Bc.shape == (V, r)
        path = np.empty((R, B - 1), np.int32)
        score = np.empty((R, B - 1), np.float32)
        margin = np.empty((R, B - 1), np.float64)
        status = np.zeros((1,), np.int32)
        self._check(self.lib.df2o_selector_walk(_p(anchors), R, B, _p(ids), _p(vals), _p(G), _p(A),
                                                _p(Bc), V, K, r, _p(path), _p(score), _p(margin),
                                                _p(status)))
        return path, score, margin, int(status[0])

    def pair_scores(self, pred, ids, vals, G, A, Bc):
        """pred [P], ids/vals [P,K], G [P,r]; returns (scores [P,K], status)."""
        pred = _c(pred, np.int32)
        ids, vals, G = _c(ids, np.int32), _c(vals, np.float32), _c(G, np.float32)
        A, Bc = _c(A, np.uint16), _c(Bc, np.uint16)
        P = pred.shape[0]
        K = ids.shape[-1]
        V, r = A.shape
        assert ids.size == P * K and G.size == P * r and Bc.shape == (V, r)
        scores = np.empty((P, K), np.float32)
        status = np.zeros((1,), np.int32)
        self._check(self.lib.df2o_selector_pair_scores(_p(pred), P, _p(ids), _p(vals), _p(G), _p(A),
                                                       _p(Bc), V, K, r, _p(scores), _p(status)))
        return scores, int(status[0])

    def selector_ce(self, scores, ids, targets, V):
        """scores/ids [P,K], targets [P]; returns (loss [P] f32, label_idx [P] int32, status)."""
        scores, ids, targets = _c(scores, np.float32), _c(ids, np.int32), _c(targets, np.int32)
        P = targets.shape[0]
        K = ids.shape[-1]
        assert ids.size == P * K and scores.size == P * K
        loss = np.empty((P,), np.float32)
        label = np.empty((P,), np.int32)
        status = np.zeros((1,), np.int32)
        self._check(self.lib.df2o_selector_ce(_p(scores), _p(ids), _p(targets), P, K, int(V), _p(loss),
                                              _p(label), _p(status)))
        return loss, label, int(status[0])

    def lattice(self, anchors, ids, vals, G, A, Bc, block_size):
        """ids/vals [R*B, K], G [R*B, r]; returns (lattice [R, B-1, K, K] f32, status)."""
        anchors = _c(anchors, np.int32)
        ids, vals, G = _c(ids, np.int32), _c(vals, np.float32), _c(G, np.float32)
        A, Bc = _c(A, np.uint16), _c(Bc, np.uint16)
        R = anchors.shape[0]
        B = int(block_size)
        K = ids.shape[-1]
        V, r = A.shape
        assert ids.size == R * B * K and G.size == R * B * r and Bc.shape == (V, r)
        lat = np.empty((R, B - 1, K, K), np.float32)
        status = np.zeros((1,), np.int32)
        self._check(self.lib.df2o_selector_lattice(_p(anchors), R, B, _p(ids), _p(vals), _p(G), _p(A),
                                                   _p(Bc), V, K, r, _p(lat), _p(status)))
        return lat, int(status[0])

    def lattice_walk(self, lattice, ids, block_size, V, uniforms=None, temperature=1.0):
        """lattice [R, B-1, K, K], ids [R*B, K], uniforms [R, B-1] or None (greedy);
        returns (path [R,B-1], score [R,B-1], margin [R,B-1], status)."""
        lattice = _c(lattice, np.float32)
        ids = _c(ids, np.int32)
        R, T, K, K2 = lattice.shape
        B = int(block_size)
        assert K == K2 and T == B - 1 and ids.size == R * B * K
        if uniforms is not None:
            uniforms = _c(uniforms, np.float32)
            assert uniforms.size == R * T
        path = np.empty((R, T), np.int32)
        score = np.empty((R, T), np.float32)
        margin = np.empty((R, T), np.float64)
        status = np.zeros((1,), np.int32)
        self._check(self.lib.df2o_lattice_walk(_p(lattice), _p(ids), R, B, K, int(V),
                                               _p(uniforms),
                                               float(temperature), _p(path), _p(score), _p(margin),
                                               _p(status)))
        return path, score, margin, int(status[0])

    # -- conv -----------------------------------------------------------------
    def conv_prepare(self, x, block_size, taps, group, W_proj, base):
        """x [P,C] uint16 (bf16) or float32; returns (y like x, dyn_out [P,taps,G] f32)."""
        x = np.ascontiguousarray(x)
        is_f32 = x.dtype == np.float32
        if not is_f32:
            x = _c(x, np.uint16)
        W_proj, base = _c(W_proj, np.uint16), _c(base, np.float32)
        P, C = x.shape
        G = C // group
        y = np.empty_like(x)
        dyn = np.empty((P, taps, G), np.float32)
        self._check(self.lib.df2o_conv_prepare(_p(x), int(is_f32), P, C, int(block_size), int(taps),
                                               int(group), _p(W_proj), _p(base), _p(y), _p(dyn)))
        return y, dyn

    def conv_finish(self, z, block_size, taps, group, dyn_out, base):
        z = np.ascontiguousarray(z)
        is_f32 = z.dtype == np.float32
        if not is_f32:
            z = _c(z, np.uint16)
        dyn_out, base = _c(dyn_out, np.float32), _c(base, np.float32)
        P, C = z.shape
        y = np.empty_like(z)
        self._check(self.lib.df2o_conv_finish(_p(z), int(is_f32), P, C, int(block_size), int(taps),
                                              int(group), _p(dyn_out), _p(base), _p(y)))
        return y

    def conv_finish_prepare(self, z, block_size, taps, group, dyn_out, base, W_proj, base_next,
                            residual=None):
        """finish(z) (+ residual), then the next prepare; returns (h, y_next, dyn_next [P,taps,G])."""
        z = np.ascontiguousarray(z)
        is_f32 = z.dtype == np.float32
        z = _c(z, np.float32 if is_f32 else np.uint16)
        if residual is not None:
            residual = _c(residual, z.dtype)
            assert residual.shape == z.shape
        dyn_out, base = _c(dyn_out, np.float32), _c(base, np.float32)
        W_proj, base_next = _c(W_proj, np.uint16), _c(base_next, np.float32)
        P, C = z.shape
        G = C // group
        h, y = np.empty_like(z), np.empty_like(z)
        dyn = np.empty((P, taps, G), np.float32)
        self._check(self.lib.df2o_conv_finish_prepare(_p(z), int(is_f32), P, C, int(block_size), int(taps),
                                                      int(group), _p(dyn_out), _p(base), _p(residual), _p(h),
                                                      _p(W_proj), _p(base_next), _p(y), _p(dyn)))
        return h, y, dyn


def default() -> Oracle:
    """The oracle built from ``dflash2_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default
