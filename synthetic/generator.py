"""Seeded, counter-based synthetic inputs for the ChunkKV workloads.

This module holds no part of the compression method: it only produces the
query window, key and value tensors (and the positions of planted "needle"
spans) that both the CUDA library and the CPU oracle consume.  Every value is a
pure function of (workload seed, layer, tensor, element index), so any slice of
any layer can be regenerated on its own, on the CPU or on a GPU, with identical
bits.

Random bits come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014): the i-th output of a stream
with key s is mix(s + (i + 1) * 0x9E3779B97F4A7C15), where mix is the
published three-step xor-shift/multiply finaliser.

Normal deviates are drawn by inverse-CDF table lookup: the top 16 bits of a
SplitMix64 output index a table of the 65536 equiprobable quantiles
Phi^-1((i + 0.5) / 65536), rounded once to fp32.  The lookup, the per-channel
scale (an exact fp64 affine map of 24 random bits, rounded once to fp32), one
IEEE fp32 multiply and one round-to-nearest-even conversion to bf16 are all
exactly specified operations, so the CPU and CUDA builds of torch produce the
same bytes.
"""
from __future__ import annotations

import math
import statistics
from dataclasses import dataclass, field

import numpy as np
import torch

GOLDEN = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1


def _to_i64(x: int) -> int:
    """Two's-complement view of an unsigned 64-bit integer."""
    x &= MASK64
    return x - (1 << 64) if x >= (1 << 63) else x


def mix64_int(z: int) -> int:
    """SplitMix64 output finaliser on a Python int (reference form)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def splitmix64_int(key: int, i: int) -> int:
    """i-th output (i >= 0) of the SplitMix64 stream with state key."""
    return mix64_int(key + (i + 1) * GOLDEN)


def _lsr(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 lanes holding unsigned 64-bit values."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def splitmix64_torch(key: int, idx: torch.Tensor) -> torch.Tensor:
    """SplitMix64 outputs for int64 counters idx (wrapping int64 arithmetic)."""
    z = idx * _to_i64(GOLDEN) + _to_i64(key + GOLDEN)
    z = (z ^ _lsr(z, 30)) * _to_i64(MIX1)
    z = (z ^ _lsr(z, 27)) * _to_i64(MIX2)
    return z ^ _lsr(z, 31)


def stream_key(*tags: int) -> int:
    """Derive an independent stream key from a tuple of small integer tags."""
    k = 0x5EED_C4A1_2024_0001
    for t in tags:
        k = mix64_int(k ^ (t & MASK64)) ^ ((k << 1) & MASK64)
        k = mix64_int(k + GOLDEN)
    return k


class HostStream:
    """Sequential SplitMix64 stream for the few host-side draws (lengths, offsets)."""

    def __init__(self, key: int):
        self.key = key & MASK64
        self.i = 0

    def next(self) -> int:
        v = splitmix64_int(self.key, self.i)
        self.i += 1
        return v

    def randint(self, lo: int, hi: int) -> int:
        """Integer in [lo, hi] (inclusive)."""
        assert hi >= lo
        return lo + self.next() % (hi - lo + 1)


_NORMAL_TABLE: dict[str, torch.Tensor] = {}


def normal_table(device) -> torch.Tensor:
    """The 65536 equiprobable N(0,1) quantiles as fp32, cached per device."""
    key = str(device)
    if key not in _NORMAL_TABLE:
        nd = statistics.NormalDist()
        vals = np.array([nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)],
                        dtype=np.float64).astype(np.float32)
        _NORMAL_TABLE[key] = torch.from_numpy(vals).to(device)
    return _NORMAL_TABLE[key]


def normal_f32(key: int, n: int, device, start: int = 0) -> torch.Tensor:
    """n standard-normal fp32 deviates, elements start..start+n-1 of stream key."""
    out = torch.empty(n, dtype=torch.float32, device=device)
    table = normal_table(device)
    step = 1 << 24
    for o in range(0, n, step):
        m = min(step, n - o)
        idx = torch.arange(start + o, start + o + m, dtype=torch.int64, device=device)
        z = splitmix64_torch(key, idx)
        out[o:o + m] = table[_lsr(z, 48)]
    return out


def uniform_scale_f32(key: int, n: int, lo: float, hi: float, device) -> torch.Tensor:
    """n values lo + (hi - lo) * u with u = 24 random bits / 2^24 (exact in fp64)."""
    idx = torch.arange(n, dtype=torch.int64, device=device)
    u24 = _lsr(splitmix64_torch(key, idx), 40).to(torch.float64)
    return (lo + (hi - lo) * (u24 / float(1 << 24))).to(torch.float32)


TENSOR_Q, TENSOR_K, TENSOR_V = 1, 2, 3
TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass
class NeedleSpec:
    """How needle keys are planted (all positions fall below the recent window)."""
    kind: str = "none"          # "none" | "chunk" | "spans"
    count: int = 0              # spans per (layer, sequence); 1 planted chunk for "chunk"
    min_len: int = 5
    max_len: int = 40
    keep_across_layers: int = 0  # spans of layer l kept by layer l+1 (rest redrawn)
    strength: float = 3.0       # needle key = strength * sqrt(d) * unit(mean window query)


@dataclass
class Workload:
    """One synthetic workload: shapes, hyper-parameters and generation recipe."""
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    seqlens: tuple
    dtype: str
    w: int
    c: int
    L_max: int
    n_layers: int
    n_reuse: int
    seed: int
    channel_scale: bool = False
    needles: NeedleSpec = field(default_factory=NeedleSpec)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def cu_seqlens(self) -> list:
        cu = [0]
        for t in self.seqlens:
            cu.append(cu[-1] + int(t))
        return cu

    @property
    def T_total(self) -> int:
        return int(sum(self.seqlens))

    def with_params(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


def gen_q_window(wl: Workload, layer: int, device) -> torch.Tensor:
    """Q_w for one layer: [B, w, Hq, d], N(0,1) in the workload dtype."""
    n = wl.B * wl.w * wl.Hq * wl.d
    x = normal_f32(stream_key(wl.seed, layer, TENSOR_Q), n, device)
    return x.view(wl.B, wl.w, wl.Hq, wl.d).to(TORCH_DTYPE[wl.dtype])


def gen_kv_raw(wl: Workload, layer: int, tensor: int, device) -> torch.Tensor:
    """K or V for one layer before needle planting: [T_total, Hkv, d]."""
    n = wl.T_total * wl.Hkv * wl.d
    x = normal_f32(stream_key(wl.seed, layer, tensor), n, device).view(wl.T_total, wl.Hkv, wl.d)
    if wl.channel_scale:
        s = uniform_scale_f32(stream_key(wl.seed, layer, tensor, 77), wl.Hkv * wl.d, 0.5, 2.0, device)
        x = x * s.view(1, wl.Hkv, wl.d)
    return x.to(TORCH_DTYPE[wl.dtype])


def _draw_spans(rs: HostStream, T: int, limit: int, count: int, lo: int, hi: int,
                taken: list) -> list:
    """Draw non-overlapping spans [s, s+L) with L in [lo, hi] and s + L <= limit."""
    spans = list(taken)
    out = []
    tries = 0
    while len(out) < count:
        tries += 1
        if tries > 100000:
            raise RuntimeError("cannot place needle spans")
        L = rs.randint(lo, hi)
        if limit - L < 0:
            continue
        s = rs.randint(0, limit - L)
        if any(s < e and a < s + L for a, e in spans):
            continue
        spans.append((s, s + L))
        out.append((s, s + L))
    return out


def needle_spans(wl: Workload) -> list:
    """Per layer, per sequence: list of (start, end) needle spans (sequence-local)."""
    ns = wl.needles
    result = []
    rs = HostStream(stream_key(wl.seed, 999))
    prev = None
    for layer in range(wl.n_layers):
        per_seq = []
        for b, T in enumerate(wl.seqlens):
            limit = max(0, T - wl.w)
            if ns.kind == "none" or limit <= 0:
                per_seq.append([])
            elif ns.kind == "chunk":
                n_full = limit // wl.c
                if n_full <= 0:
                    per_seq.append([])
                    continue
                i = rs.randint(0, n_full - 1)
                per_seq.append([(i * wl.c, i * wl.c + wl.c)])
            else:
                keep = []
                if prev is not None and ns.keep_across_layers > 0:
                    old = list(prev[b])
                    # seeded choice of which spans survive into this layer
                    for _ in range(min(ns.keep_across_layers, len(old))):
                        keep.append(old.pop(rs.randint(0, len(old) - 1)))
                new = _draw_spans(rs, T, limit, ns.count - len(keep), ns.min_len,
                                  min(ns.max_len, limit), keep)
                per_seq.append(sorted(keep + new))
        result.append(per_seq)
        prev = per_seq
    return result


def needle_vectors(wl: Workload, q_win: torch.Tensor) -> np.ndarray:
    """Per (sequence, kv head): strength * sqrt(d) * unit(mean of the group's window queries).

    Returned in fp64 [B, Hkv, d]; the caller rounds to the workload dtype.
    """
    q = q_win.detach().to("cpu", torch.float64).numpy()      # [B, w, Hq, d]
    B, w, Hq, d = q.shape
    G = Hq // wl.Hkv
    qg = q.reshape(B, w, wl.Hkv, G, d)
    mean = qg.mean(axis=(1, 3))                              # [B, Hkv, d]
    norm = np.sqrt((mean * mean).sum(axis=-1, keepdims=True))
    norm[norm == 0] = 1.0
    return wl.needles.strength * math.sqrt(d) * mean / norm


def make_layer(wl: Workload, layer: int, device, spans=None, with_q=None):
    """Generate (q_win or None, k, v) for one layer, needles planted into K.

    q_win is produced for every layer that scores under index reuse (layer %
    n_reuse == 0) unless with_q overrides; needle keys of a reuse layer follow
    the query window of its own layer index, which is generated (but not
    returned) when needed.
    """
    if spans is None:
        spans = needle_spans(wl)[layer]
    scoring = (layer % wl.n_reuse == 0) if with_q is None else with_q
    q = gen_q_window(wl, layer, device)
    k = gen_kv_raw(wl, layer, TENSOR_K, device)
    v = gen_kv_raw(wl, layer, TENSOR_V, device)
    if wl.w > 0 and any(len(s) for s in spans):         # needles follow the window queries
        vec = torch.from_numpy(needle_vectors(wl, q)).to(TORCH_DTYPE[wl.dtype]).to(device)
        cu = wl.cu_seqlens
        for b, seq_spans in enumerate(spans):
            for (s, e) in seq_spans:
                k[cu[b] + s: cu[b] + e] = vec[b].unsqueeze(0)
    return (q if scoring else None), k, v


def make_all_layers(wl: Workload, device):
    """All layers: lists q_win (None for reuse layers), k, v, plus the needle spans."""
    spans = needle_spans(wl)
    qs, ks, vs = [], [], []
    for layer in range(wl.n_layers):
        q, k, v = make_layer(wl, layer, device, spans=spans[layer])
        qs.append(q)
        ks.append(k)
        vs.append(v)
    return qs, ks, vs, spans
