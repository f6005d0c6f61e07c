"""Workload definitions and seeded tensor draws.

Each workload is a THD pack (segments concatenated along the token axis,
described by ``cu_seqlens``) plus one or two attention layers. The five
named packs are the sizes this library is measured and checked on:

* ``tiny``       256 tokens in segments [100, 37, 119]; H=4, indexer 4x64,
                 cmp_ratio 4, topk 8, window 16.
* ``prefill4k``  4096 tokens in 8 lognormal segments (median 400); H=64,
                 indexer 64x128, cmp_ratio 4, topk 512, window 128.
* ``long16k``    16384 tokens in one segment; same layer as ``prefill4k``.
* ``hca32k``     32768 tokens in 16 lognormal segments (median 2000);
                 compressor-only layer (no indexer), cmp_ratio 128.
* ``mixed32k``   32768 tokens in 64 lognormal segments (median 400, lengths
                 1..4000, one segment of length 1 and one of length 3);
                 a cmp_ratio-4 indexer layer followed by a cmp_ratio-128
                 compressor-only layer.

Segment-length recipe (a reading: only the median is fixed for the
lognormal packs). Draw ``n`` lengths from a lognormal with ``mu = ln(median)``
and ``sigma = sqrt(2 ln((T/n)/median))`` so that the mean is ``T/n``; scale
to the token budget and floor; clamp to ``>= 1`` (and to the pack's maximum);
replace multiples of 4 by ``L - 1``; then repair the sum by round-robin
``+-1`` steps that skip any result divisible by 4 or below 2.
``mixed32k`` finally pins one slot to length 1 and one to length 3 before the
repair, and the repair leaves those two slots alone.

Tensor recipe: one ``torch.Generator('cpu')`` seeded with the pack's seed,
drawing, per layer and in this order, q, ori_kv, cmp_kv, q_idx, k_idx, w,
sinks. Every tensor is N(0,1) (cast to bf16 where the layer stores bf16),
except ``w`` of the tiny pack, which is U(0,1). ``cmp_kv`` and ``k_idx`` are
drawn with ``T // cmp_ratio`` rows, an upper bound on the compressed row
count; the caller keeps the leading rows it needs.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

_CHUNK = 1 << 24  # elements per draw: bounds the fp32 temporary


@dataclass(frozen=True)
class LayerSpec:
    cmp_ratio: int
    indexer: bool            # True: lightning indexer + top-k; False: compressor-only (HCA)
    topk: int = 0            # indexer layers only
    index_heads: int = 0     # Hi
    index_dim: int = 0       # Di


@dataclass(frozen=True)
class PackSpec:
    name: str
    lengths: tuple
    heads: int               # H
    dim: int                 # D (= d_v; K and V share the row)
    win_left: int            # window = win_left + 1 rows, self included
    layers: tuple
    seed: int
    w_uniform: bool = False
    softmax_scale: float = field(default=0.0)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale else 1.0 / math.sqrt(self.dim)


def lognormal_lengths(seed: int, total: int, n: int, median: float,
                      max_len: int | None = None, pin_short: bool = False) -> list:
    """Segment lengths summing to ``total``; see the module docstring."""
    sigma = math.sqrt(2.0 * math.log((total / n) / median))
    raw = np.random.default_rng(seed).lognormal(math.log(median), sigma, n)
    lens = np.floor(raw * total / raw.sum()).astype(np.int64)
    lens = np.maximum(lens, 1)
    if max_len is not None:
        lens = np.minimum(lens, max_len)
    lens = np.where(lens % 4 == 0, lens - 1, lens)
    frozen = set()
    if pin_short:
        a, b = n // 3, (2 * n) // 3
        lens[a], lens[b] = 1, 3
        frozen = {a, b}
    lens = [int(x) for x in lens]
    deficit = total - sum(lens)
    guard = 0
    jump = False  # after a pass with no legal +-1 move, allow +-2 steps over a multiple of 4
    while deficit != 0:
        step = 1 if deficit > 0 else -1
        moved = False
        for i in range(n):
            if deficit == 0:
                break
            if i in frozen:
                continue
            nxt = lens[i] + step
            if nxt % 4 == 0:
                if not jump or abs(deficit) < 2:
                    continue
                nxt += step
            if nxt < 2 or (max_len is not None and nxt > max_len):
                continue
            deficit -= nxt - lens[i]
            lens[i] = nxt
            moved = True
        guard += 1
        if not moved:
            if jump:
                raise RuntimeError("length repair did not converge")
            jump = True
        else:
            jump = False
        if guard > 100000:
            raise RuntimeError("length repair did not converge")
    return lens


def make_cu_seqlens(lengths) -> torch.Tensor:
    """int32 prefix sums ``[0, l0, l0+l1, ...]`` (the THD packing format)."""
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return torch.from_numpy(cu.astype(np.int32))


def _indexer_layer(r=4, k=512, hi=64, di=128):
    return LayerSpec(cmp_ratio=r, indexer=True, topk=k, index_heads=hi, index_dim=di)


def _hca_layer(r=128):
    return LayerSpec(cmp_ratio=r, indexer=False)


def pack_spec(name: str) -> PackSpec:
    if name == "tiny":
        return PackSpec("tiny", (100, 37, 119), heads=4, dim=512, win_left=15,
                        layers=(_indexer_layer(4, 8, 4, 64),), seed=1, w_uniform=True)
    if name == "prefill4k":
        return PackSpec("prefill4k", tuple(lognormal_lengths(2, 4096, 8, 400)), heads=64,
                        dim=512, win_left=127, layers=(_indexer_layer(),), seed=2)
    if name == "long16k":
        return PackSpec("long16k", (16384,), heads=64, dim=512, win_left=127,
                        layers=(_indexer_layer(),), seed=3)
    if name == "hca32k":
        return PackSpec("hca32k", tuple(lognormal_lengths(4, 32768, 16, 2000)), heads=64,
                        dim=512, win_left=127, layers=(_hca_layer(),), seed=4)
    if name == "mixed32k":
        return PackSpec("mixed32k",
                        tuple(lognormal_lengths(5, 32768, 64, 400, max_len=4000, pin_short=True)),
                        heads=64, dim=512, win_left=127,
                        layers=(_indexer_layer(), _hca_layer()), seed=5)
    raise KeyError(name)


CONFIGS = ("tiny", "prefill4k", "long16k", "hca32k", "mixed32k")


def _randn(gen: torch.Generator, shape, dtype) -> torch.Tensor:
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=dtype)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        out[s:e] = torch.randn(e - s, generator=gen, dtype=torch.float32).to(dtype)
    return out.view(*shape)


def _rand(gen: torch.Generator, shape) -> torch.Tensor:
    return torch.rand(*shape, generator=gen, dtype=torch.float32)


def draw_layer_tensors(spec: PackSpec, gen: torch.Generator, layer: LayerSpec) -> dict:
    """Draw one layer's tensors (CPU) from ``gen`` in the fixed order."""
    T, H, D = spec.total_tokens, spec.heads, spec.dim
    rows_c = max(T // layer.cmp_ratio, 0)
    bf16 = torch.bfloat16
    out = {}
    out["q"] = _randn(gen, (T, H, D), bf16)
    out["ori_kv"] = _randn(gen, (T, D), bf16)
    out["cmp_kv"] = _randn(gen, (rows_c, D), bf16)
    if layer.indexer:
        hi, di = layer.index_heads, layer.index_dim
        out["q_idx"] = _randn(gen, (T, hi, di), bf16)
        out["k_idx"] = _randn(gen, (rows_c, di), bf16)
        out["w"] = _rand(gen, (T, hi)) if spec.w_uniform else _randn(gen, (T, hi), torch.float32)
    out["sinks"] = _randn(gen, (H,), torch.float32)
    return out


def draw_pack(spec: PackSpec) -> list:
    """All layers of a pack, in order, from one generator seeded with ``spec.seed``."""
    gen = torch.Generator("cpu").manual_seed(spec.seed)
    return [draw_layer_tensors(spec, gen, layer) for layer in spec.layers]


def draw_indexer_tensors(total_tokens: int, rows_c: int, index_heads: int, index_dim: int,
                         seed: int, w_uniform: bool = False) -> dict:
    """Indexer inputs alone (CPU): q_idx [T, Hi, Di] and k_idx [rows_c, Di] bf16
    N(0,1), w [T, Hi] fp32 (N(0,1), or U(0,1) with ``w_uniform``), drawn in that
    order from one generator seeded with ``seed``."""
    gen = torch.Generator("cpu").manual_seed(seed)
    bf16 = torch.bfloat16
    out = {"q_idx": _randn(gen, (total_tokens, index_heads, index_dim), bf16),
           "k_idx": _randn(gen, (rows_c, index_dim), bf16)}
    out["w"] = (_rand(gen, (total_tokens, index_heads)) if w_uniform
                else _randn(gen, (total_tokens, index_heads), torch.float32))
    return out


def draw_uniform(shape, seed: int, low: float = 0.0, high: float = 1.0) -> torch.Tensor:
    """fp32 U(low, high) tensor (CPU) from a generator seeded with ``seed``."""
    gen = torch.Generator("cpu").manual_seed(seed)
    return low + (high - low) * _rand(gen, tuple(shape))


def draw_normal(shape, seed: int) -> torch.Tensor:
    """fp32 N(0,1) tensor (CPU) from a generator seeded with ``seed``."""
    gen = torch.Generator("cpu").manual_seed(seed)
    return _randn(gen, tuple(shape), torch.float32)
