"""Seeded synthetic workloads for the DFlash2 draft-block head.

This module only draws inputs: it holds none of the method's arithmetic, and it
is the one piece shared by the CUDA path's tests/bench and the CPU oracle.  Every
tensor comes from its own counter-derived PCG64 stream (seed, tensor tag), so
changing one tensor's shape never shifts another's values.

bf16 tensors are returned as ``uint16`` arrays of raw bfloat16 bit patterns,
drawn in fp32 and rounded to nearest-even; both sides therefore read exactly the
same bf16 values.  Shapes and value distributions follow the five workloads of
the draft-block head:

=========  =====================================================================
tiny       V 4096, D 256, r 32, K 4, block 8 (anchor + 7 drafted), 2 requests;
           conv taps 2, group 16; fp32 draws ~N(0, 0.02) for every tensor, head
           operands rounded to bf16, conv activations kept fp32
batch1     Qwen3-8B-shaped batch-1 latency: D 4096, V 151936, r 256, K 16,
           block 8, 1 request; weights ~N(0, 0.02), hidden ~N(0, 1), bf16
batched    27B-drafter-shaped serving: D 5120, V 248320, r 256, K 16, block 8,
           64 requests (512 positions)
conv       training-packed conv: 4 sequences x 512 anchor blocks x block 8,
           C 5120, taps 2, group 16; base tap 0 ~N(1, 0.1), later taps ~N(0, 0.1)
stress     D 4096, V 151936, r 512, K 64, block 16, 256 requests (4096
           positions), conv taps 4; ~30% of rows planted with a near-tie at
           rank K (a near-duplicate pair of W_lm rows placed at ranks K, K+1)
=========  =====================================================================

No public dataset, benchmark suite or trained checkpoint is used or imitated:
the pages' accuracy numbers come from such data, and these synthetic draws only
stand in for the tensor shapes and magnitudes those workloads have.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import os
import zlib

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    V: int          # verifier vocabulary
    D: int          # hidden size (= conv channels C)
    r: int          # selector rank
    K: int          # selector top-K
    B: int          # block size (anchor + B-1 drafted positions)
    R: int          # requests (anchor blocks)
    taps: int       # conv taps
    g: int          # conv group size
    act: str        # conv activation dtype: "f32" or "bf16"
    h_std: float    # hidden-state scale
    w_std: float = 0.02
    near_tie_frac: float = 0.0
    conv_only: bool = False
    seed: int = 0

    @property
    def P(self) -> int:
        return self.R * self.B

    @property
    def C(self) -> int:
        return self.D

    @property
    def G(self) -> int:
        return self.D // self.g

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


TINY = Workload("tiny", V=4096, D=256, r=32, K=4, B=8, R=2, taps=2, g=16, act="f32",
                h_std=0.02, seed=0)
BATCH1 = Workload("batch1", V=151936, D=4096, r=256, K=16, B=8, R=1, taps=2, g=16, act="bf16",
                  h_std=1.0, seed=1)
BATCHED = Workload("batched", V=248320, D=5120, r=256, K=16, B=8, R=64, taps=2, g=16, act="bf16",
                   h_std=1.0, seed=2)
CONV_PACKED = Workload("conv", V=0, D=5120, r=0, K=0, B=8, R=4 * 512, taps=2, g=16, act="bf16",
                       h_std=1.0, conv_only=True, seed=3)
STRESS = Workload("stress", V=151936, D=4096, r=512, K=64, B=16, R=256, taps=4, g=16, act="bf16",
                  h_std=1.0, near_tie_frac=0.30, seed=4)

CONFIGS = [TINY, BATCH1, BATCHED, CONV_PACKED, STRESS]
BY_NAME = {w.name: w for w in CONFIGS}


# ----------------------------------------------------------------- drawing --

def _gen(seed: int, tag: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, zlib.crc32(tag.encode())])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bfloat16 (nearest-even) and return the bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact fp32 value of bfloat16 bit patterns."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_CHUNK = 1 << 22


def normal_bf16(seed: int, tag: str, shape, std: float, mean: float = 0.0) -> np.ndarray:
    """N(mean, std^2) draws rounded to bf16.  Chunk c of 2^22 elements comes from
    its own stream (seed, tag, c), so the values do not depend on how many host
    threads fill them."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    key = zlib.crc32(tag.encode())

    def fill(c):
        s = c * _CHUNK
        e = min(n, s + _CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, key, c])))
        v = g.standard_normal(e - s, dtype=np.float32)
        v *= np.float32(std)
        if mean:
            v += np.float32(mean)
        out[s:e] = f32_to_bf16_bits(v)

    nchunks = (n + _CHUNK - 1) // _CHUNK
    if nchunks <= 1:
        for c in range(nchunks):
            fill(c)
    else:
        with concurrent.futures.ThreadPoolExecutor(min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def normal_f32(seed: int, tag: str, shape, std: float, mean: float = 0.0) -> np.ndarray:
    g = _gen(seed, tag)
    v = g.standard_normal(int(np.prod(shape)), dtype=np.float32) * np.float32(std)
    if mean:
        v += np.float32(mean)
    return v.reshape(shape)


def uniform_ids(seed: int, tag: str, n: int, V: int) -> np.ndarray:
    return _gen(seed, tag).integers(0, V, size=n, dtype=np.int64).astype(np.int32)


# ----------------------------------------------------------------- inputs --

def head_inputs(w: Workload, selector_std: float | None = None, rows: int | None = None) -> dict:
    """Inputs of the head: h [P,D], W_lm [V,D], W_H [r,D], A/Bc [V,r] (bf16 bits),
    anchors [R] and teacher-forcing predecessors pred [P] (int32).

    ``selector_std`` overrides the codebooks' scale (a "strong selector" whose
    transition term is comparable to the unary logits).  ``rows`` limits h to its
    first rows (for oracle-sized slices of a large workload)."""
    assert not w.conv_only
    s = w.seed
    P = w.P if rows is None else rows
    A, Bc = selector_codebooks(w, selector_std)
    out = {
        "W_lm": normal_bf16(s, "W_lm", (w.V, w.D), w.w_std),
        "W_H": normal_bf16(s, "W_H", (w.r, w.D), w.w_std),
        "A": A,
        "Bc": Bc,
        "anchors": uniform_ids(s, "anchors", w.R, w.V),
        "pred": uniform_ids(s, "pred", w.P, w.V),
    }
    if w.near_tie_frac > 0:
        h, spiked = _near_tie_hidden(w, out["W_lm"])
        out["h"] = h
        out["spiked_rows"] = spiked
    else:
        out["h"] = normal_bf16(s, "h", (w.P, w.D), w.h_std)
        out["spiked_rows"] = np.zeros(0, np.int64)
    if rows is not None:
        out["h"] = out["h"][:rows]
        out["pred"] = out["pred"][:rows]
    return out


def selector_codebooks(w: Workload, selector_std: float | None = None):
    """The predecessor and successor codebooks A, Bc [V, r] (bf16 bits), at the
    workload's weight scale or at ``selector_std`` (the "strong selector")."""
    cb_std = w.w_std if selector_std is None else selector_std
    return (normal_bf16(w.seed, "A", (w.V, w.r), cb_std), normal_bf16(w.seed, "B", (w.V, w.r), cb_std))


def conv_inputs(w: Workload) -> dict:
    """Inputs of the conv: x, z [P,C] (fp32 or bf16 bits), W_proj [2*taps*G, C]
    (bf16 bits), base [2, taps, C] (fp32)."""
    s = w.seed
    P, C = w.P, w.C
    nproj = 2 * w.taps * w.G
    if w.act == "f32":
        x = normal_f32(s, "conv_x", (P, C), w.h_std)
        z = normal_f32(s, "conv_z", (P, C), w.h_std)
        base = normal_f32(s, "conv_base", (2, w.taps, C), 0.02)
    else:
        x = normal_bf16(s, "conv_x", (P, C), 1.0)
        z = normal_bf16(s, "conv_z", (P, C), 1.0)
        base = normal_f32(s, "conv_base", (2, w.taps, C), 0.1)
        base[:, 0, :] += np.float32(1.0)
    W_proj = normal_bf16(s, "conv_W_proj", (nproj, C), w.w_std)
    return {"x": x, "z": z, "W_proj": W_proj, "base": base}


def _near_tie_hidden(w: Workload, W_lm: np.ndarray):
    """Plant near-ties at rank K in a fraction of rows (modifies W_lm in place).

    A pool of disjoint pairs (v, v') is drawn; W_lm[v'] becomes a copy of W_lm[v]
    (a quarter of the pairs exactly, the rest with 1-3 coordinates moved by one
    bf16 step), so U(v) and U(v') differ by ~1e-4 or not at all.  A spiked row gets
    h = z + s * W_lm[v] / |W_lm[v]|, with s chosen so that exactly K-1 other tokens
    stay above v: v and v' then sit at ranks K and K+1.  The other rows keep
    h = z ~ N(0, 1)."""
    s = w.seed
    g = _gen(s, "near_tie")
    P, V, D, K = w.P, w.V, w.D, w.K
    z = normal_f32(s, "h", (P, D), w.h_std)
    n_spiked = int(round(w.near_tie_frac * P))
    rows = np.sort(g.choice(P, size=n_spiked, replace=False))
    n_pairs = min(2048, n_spiked) if n_spiked else 0
    pool = g.choice(V, size=2 * n_pairs, replace=False)
    vs, v2s = pool[:n_pairs], pool[n_pairs:]
    for i in range(n_pairs):
        W_lm[v2s[i]] = W_lm[vs[i]]
        if i % 4:
            cols = g.choice(D, size=1 + i % 3, replace=False)
            step = np.where(g.random(cols.size) < 0.5, 1, -1).astype(np.int32)
            bits = W_lm[v2s[i], cols].astype(np.int32)
            W_lm[v2s[i], cols] = np.clip(bits + step, 0, 0xFFFF).astype(np.uint16)
    which = g.integers(0, max(n_pairs, 1), size=n_spiked)
    h = z.copy()
    # Background logits U_z = W z and alignments c = W w_hat_v, in chunks of W rows.
    Wf_rows = 16384
    if n_spiked:
        vsel = vs[which]
        wv = bf16_bits_to_f32(W_lm[vsel])
        wv_hat = wv / np.linalg.norm(wv, axis=1, keepdims=True)
        M = np.concatenate([z[rows], wv_hat], axis=0).T.astype(np.float32)  # [D, 2n]
        Uz = np.empty((n_spiked, V), np.float32)
        Cw = np.empty((n_spiked, V), np.float32)
        for a in range(0, V, Wf_rows):
            b = min(V, a + Wf_rows)
            prod = bf16_bits_to_f32(W_lm[a:b]) @ M
            Uz[:, a:b] = prod[:, :n_spiked].T
            Cw[:, a:b] = prod[:, n_spiked:].T
        for k, p in enumerate(rows):
            v, v2 = vsel[k], v2s[which[k]]
            cv = Cw[k, v]
            with np.errstate(divide="ignore", invalid="ignore"):
                sx = (Uz[k] - Uz[k, v]) / (cv - Cw[k])
            sx[v] = -np.inf
            sx[v2] = -np.inf
            # s between the (K-1)-th and K-th largest crossing points
            top = np.partition(sx, V - K)[V - K:]
            top.sort()
            s_hi, s_lo = top[1], top[0]
            sv = 0.5 * (s_hi + s_lo) if np.isfinite(s_lo) else s_hi + 1.0
            h[p] = z[p] + np.float32(max(sv, 0.0)) * wv_hat[k]
    return f32_to_bf16_bits(h), rows.astype(np.int64)
