"""Seeded synthetic inputs for one TwoTower denoiser step.

This module only *draws* inputs: query/key/value tensors, paged context KV
caches with shuffled page order, block KV, vocabulary logits, and the clean
tokens, uniform draws and diffusion times of the training-side corruption.  It contains
none of the step's arithmetic (no attention, no softmax, no unmasking rule), so
that the float64 oracle and the CUDA path can both consume the very same values
without sharing any of the code under test.

Recipe (the pages fix no weights or data, so every tensor is synthetic):

* Q, K, V ~ N(0, 1) * ``qkv_scale`` (1/sqrt(head_dim) by default), drawn in
  float32 and rounded to bfloat16 with round-to-nearest-even (``bf16_bits``).
  The denoiser's queries attend to the frozen context tower's per-layer KV and
  to the block's own KV (TwoTower summary, gist.science/de, "Technisches
  Resümee — Architektur").
* Logits ~ N(0, 3) (standard deviation 3) plus a planted peak of height
  U[0, ``peak_hi``] added at one uniformly drawn token per block position.
* The context KV lives in pages of ``page_size`` tokens.  Every sequence owns
  ``max_pages_per_seq`` pages taken from a random permutation of the pool, so
  logical order and physical order differ; a few spare pages belong to no
  sequence.  Slots past a sequence's length can be filled with garbage (NaN or
  huge values) to prove that nothing reads them.

Seeds: ``numpy.random.Generator(PCG64(SeedSequence([seed, config_id, block,
step, layer, tensor_id])))``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

# tensor ids used in the seed sequence
T_Q, T_KBLK, T_VBLK, T_KPOOL, T_VPOOL, T_LOGITS, T_PAGES, T_LENS, T_KNEW, T_VNEW, T_PLANT, \
    T_UNIFORM, T_TIME, T_CLEAN = range(14)


def rng_for(seed: int, config_id: int, block: int = 0, step: int = 0, layer: int = 0,
            tensor_id: int = 0) -> np.random.Generator:
    """A generator keyed by (seed, config, block, step, layer, tensor)."""
    ss = np.random.SeedSequence([int(seed), int(config_id), int(block), int(step), int(layer),
                                 int(tensor_id)])
    return np.random.Generator(np.random.PCG64(ss))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round-to-nearest-even); returns uint16 bit patterns."""
    x32 = np.ascontiguousarray(x, dtype=np.float32)
    u = x32.view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    out = ((u + bias) >> 16).astype(np.uint16)
    nan = np.isnan(x32)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def _normal32(rng: np.random.Generator, shape, scale: float) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x


def _encode(x32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_bits(x32)
    if dtype == "f32":
        return np.ascontiguousarray(x32, dtype=np.float32)
    raise ValueError(dtype)


@dataclasses.dataclass
class StepConfig:
    """Shapes and value distributions of one denoise-step workload."""
    name: str
    config_id: int
    B: int
    S: int
    Hq: int
    Hkv: int
    D: int
    V: int
    dtype: str                      # "bf16" or "f32"
    len_lo: int                     # context lengths ~ U[len_lo, len_hi] (inclusive)
    len_hi: int
    tau: float = 0.9
    T: int = 16
    n_layers: int = 1
    n_blocks: int = 1
    page_size: int = 64
    qkv_scale: Optional[float] = None   # None -> 1/sqrt(D)
    logit_std: float = 3.0
    peak_hi: float = 12.0

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D) if self.qkv_scale is None else self.qkv_scale

    def replace(self, **kw) -> "StepConfig":
        return dataclasses.replace(self, **kw)


# The five workloads of the hot path, plus the fixed-length 8K headline.
CONFIGS = {
    "tiny": StepConfig("tiny", 0, B=1, S=16, Hq=4, Hkv=1, D=64, V=1024, dtype="f32",
                       len_lo=64, len_hi=64, T=4),
    "single": StepConfig("single", 1, B=1, S=16, Hq=32, Hkv=2, D=128, V=131072, dtype="bf16",
                         len_lo=4096, len_hi=4096),
    "ragged": StepConfig("ragged", 2, B=32, S=16, Hq=32, Hkv=2, D=128, V=131072, dtype="bf16",
                         len_lo=1024, len_hi=8192),
    "long": StepConfig("long", 3, B=4, S=16, Hq=32, Hkv=2, D=128, V=131072, dtype="bf16",
                       len_lo=131072, len_hi=131072),
    "loop": StepConfig("loop", 4, B=16, S=16, Hq=32, Hkv=2, D=128, V=131072, dtype="bf16",
                       len_lo=16384, len_hi=16384, n_layers=6, T=16, n_blocks=8),
    "ctx8k": StepConfig("ctx8k", 5, B=32, S=16, Hq=32, Hkv=2, D=128, V=131072, dtype="bf16",
                        len_lo=8192, len_hi=8192),
}


def draw_lengths(cfg: StepConfig, seed: int = 0) -> np.ndarray:
    if cfg.len_lo == cfg.len_hi:
        return np.full(cfg.B, cfg.len_lo, dtype=np.int32)
    r = rng_for(seed, cfg.config_id, tensor_id=T_LENS)
    return r.integers(cfg.len_lo, cfg.len_hi + 1, size=cfg.B).astype(np.int32)


@dataclasses.dataclass
class PagedCache:
    """One layer's paged context cache in host memory (bit patterns for bf16)."""
    k_pool: np.ndarray              # [num_pages, Hkv, page_size, D]
    v_pool: np.ndarray
    page_table: np.ndarray          # [B, max_pages_per_seq] int32
    ctx_len: np.ndarray             # [B] int32
    page_size: int
    dtype: str

    @property
    def num_pages(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.page_table.shape[1])


def draw_page_table(cfg: StepConfig, capacity_tokens: int, seed: int = 0, spare_pages: int = 3):
    """Shuffled page ids: sequence b owns ``page_table[b]``; a few spare pages are never owned."""
    maxp = max(1, -(-capacity_tokens // cfg.page_size))
    num_pages = cfg.B * maxp + spare_pages
    r = rng_for(seed, cfg.config_id, tensor_id=T_PAGES)
    perm = r.permutation(num_pages).astype(np.int32)
    table = perm[: cfg.B * maxp].reshape(cfg.B, maxp).copy()
    return table, num_pages


def draw_paged_cache(cfg: StepConfig, lens: np.ndarray, capacity_tokens: int, seed: int = 0,
                     layer: int = 0, garbage: Optional[str] = None,
                     page_table: Optional[np.ndarray] = None,
                     num_pages: Optional[int] = None) -> PagedCache:
    """Draw one layer's K/V pools.

    ``garbage``: None keeps the drawn values everywhere; "nan" or "huge" overwrites every
    slot that is not a live context position (beyond ``lens[b]`` and in spare pages).
    """
    if page_table is None:
        page_table, num_pages = draw_page_table(cfg, capacity_tokens, seed)
    shape = (num_pages, cfg.Hkv, cfg.page_size, cfg.D)
    pools = []
    for tid in (T_KPOOL, T_VPOOL):
        r = rng_for(seed, cfg.config_id, layer=layer, tensor_id=tid)
        x = _normal32(r, shape, cfg.scale)
        if garbage is not None:
            live = np.zeros((num_pages, cfg.page_size), dtype=bool)
            for b in range(cfg.B):
                L = int(lens[b])
                full, rem = divmod(L, cfg.page_size)
                live[page_table[b, :full]] = True
                if rem:
                    live[page_table[b, full], :rem] = True
            fill = np.float32(np.nan) if garbage == "nan" else np.float32(3.0e38)
            x[np.broadcast_to((~live)[:, None, :, None], x.shape)] = fill
        pools.append(_encode(x, cfg.dtype))
    return PagedCache(pools[0], pools[1], page_table.astype(np.int32), lens.astype(np.int32).copy(),
                      cfg.page_size, cfg.dtype)


def draw_block_qkv(cfg: StepConfig, seed: int = 0, block: int = 0, step: int = 0, layer: int = 0):
    """Block queries [B,S,Hq,D] and the block's own keys/values [B,S,Hkv,D]."""
    out = []
    for tid, H in ((T_Q, cfg.Hq), (T_KBLK, cfg.Hkv), (T_VBLK, cfg.Hkv)):
        r = rng_for(seed, cfg.config_id, block, step, layer, tid)
        out.append(_encode(_normal32(r, (cfg.B, cfg.S, H, cfg.D), cfg.scale), cfg.dtype))
    return tuple(out)


def draw_new_block_kv(cfg: StepConfig, seed: int = 0, block: int = 0, layer: int = 0):
    """KV of a committed block as the context tower would produce it: seeded N(0,1) stand-ins."""
    out = []
    for tid in (T_KNEW, T_VNEW):
        r = rng_for(seed, cfg.config_id, block, 0, layer, tid)
        out.append(_encode(_normal32(r, (cfg.B, cfg.S, cfg.Hkv, cfg.D), 1.0), cfg.dtype))
    return tuple(out)


def draw_logits(cfg: StepConfig, seed: int = 0, block: int = 0, step: int = 0,
                peak_hi: Optional[float] = None, rows: Optional[int] = None) -> np.ndarray:
    """Logits [B,S,V]: N(0, logit_std) plus a peak U[0, peak_hi] at one uniform token per row."""
    peak_hi = cfg.peak_hi if peak_hi is None else peak_hi
    B = cfg.B if rows is None else rows
    r = rng_for(seed, cfg.config_id, block, step, 0, T_LOGITS)
    x = _normal32(r, (B, cfg.S, cfg.V), cfg.logit_std)
    tok = r.integers(0, cfg.V, size=(B, cfg.S))
    h = r.uniform(0.0, peak_hi, size=(B, cfg.S)).astype(np.float32)
    bi, si = np.meshgrid(np.arange(B), np.arange(cfg.S), indexing="ij")
    x[bi, si, tok] += h
    return _encode(x, cfg.dtype)


def plant_keys(cfg: StepConfig, cache: PagedCache, q: np.ndarray, seed: int = 0, per_seq: int = 4,
               boost: float = 8.0, positions: Optional[list] = None) -> list:
    """Overwrite a few context keys with a multiple of a query head's vector so that their
    scores dominate (stress variant).  Positions default to page edges, the last partial page
    and random places.  Returns the (b, position) pairs that were planted."""
    r = rng_for(seed, cfg.config_id, tensor_id=T_PLANT)
    planted = []
    for b in range(cfg.B):
        L = int(cache.ctx_len[b])
        if L == 0:
            continue
        cand = positions if positions is not None else sorted(set(
            [0, min(L - 1, cfg.page_size - 1), min(L - 1, cfg.page_size), L - 1]
            + list(r.integers(0, L, size=max(0, per_seq - 4)))))
        for j in cand:
            j = int(j)
            if not 0 <= j < L:
                continue
            g = int(r.integers(0, cfg.Hkv))
            h = g * cfg.G + int(r.integers(0, cfg.G))
            s = int(r.integers(0, cfg.S))
            page = cache.page_table[b, j // cfg.page_size]
            slot = j % cfg.page_size
            qv = _decode(q[b, s, h], cfg.dtype).astype(np.float32)
            cache.k_pool[page, g, slot] = _encode(qv * np.float32(boost), cfg.dtype)
            planted.append((b, j))
    return planted


def _decode(x: np.ndarray, dtype: str) -> np.ndarray:
    """bf16 bit patterns (or float32) -> float32; used only to build stress inputs."""
    if dtype == "bf16":
        return (x.astype(np.uint32) << 16).view(np.float32)
    return np.asarray(x, dtype=np.float32)


def draw_corruption(cfg: StepConfig, seed: int = 0, block: int = 0):
    """Inputs of the masked-diffusion corruption of one batch of clean blocks: clean tokens
    [B,S] ~ uniform over the vocabulary, uniform draws u [B,S] ~ U[0, 1) and one diffusion
    time t [B] ~ U[0, 1] per sequence (float32)."""
    clean = rng_for(seed, cfg.config_id, block, 0, 0, T_CLEAN).integers(0, cfg.V, size=(cfg.B, cfg.S))
    u = rng_for(seed, cfg.config_id, block, 0, 0, T_UNIFORM).random((cfg.B, cfg.S), dtype=np.float32)
    t = rng_for(seed, cfg.config_id, block, 0, 0, T_TIME).random(cfg.B, dtype=np.float32)
    return clean.astype(np.int32), u, t
