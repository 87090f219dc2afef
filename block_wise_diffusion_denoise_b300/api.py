"""Thin PyTorch binding of the C ABI (argument marshalling only).

Every function here checks that its tensors are contiguous CUDA tensors of the
expected dtype, passes their ``data_ptr()`` and the current CUDA stream to the
library, and raises ``TTError`` on a non-zero status.  All arithmetic of the
denoise step runs in the library's CUDA kernels; PyTorch only provides device
memory and streams.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
from typing import Optional, Sequence

import torch

from . import _native as N
from ._native import TT_BF16, TT_FP32, TTError  # noqa: F401

_DT = {torch.bfloat16: TT_BF16, torch.float32: TT_FP32}


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _need(t: Optional[torch.Tensor], name: str, dtype=None, shape=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, not on the current device cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _ws(ws: torch.Tensor):
    """(pointer, size in bytes) of a caller's workspace tensor."""
    _need(ws, "ws")
    return ws.data_ptr(), ws.numel() * ws.element_size()


def _cover(cache: "KVCache", B: int) -> None:
    """The cache's page table and lengths must cover the B sequences of the call."""
    if cache.ctx_len.shape[0] < B:
        raise ValueError(f"the cache holds {cache.ctx_len.shape[0]} sequences, the call {B}")


def _err(dev_err: Optional[torch.Tensor]) -> Optional[int]:
    _need(dev_err, "dev_err", torch.int32, allow_none=True)
    if dev_err is not None and dev_err.numel() < 1:
        raise ValueError("dev_err must hold at least one int32")
    return _ptr(dev_err)


@dataclasses.dataclass
class KVCache:
    """One attention layer's paged context KV cache (device tensors).

    k_pool, v_pool: [num_pages, Hkv, page_size, D] (bf16 or fp32);
    page_table: [B, max_pages_per_seq] int32; ctx_len: [B] int32."""
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    page_table: torch.Tensor
    ctx_len: torch.Tensor

    def __post_init__(self):
        if self.k_pool.dtype not in _DT or self.v_pool.dtype != self.k_pool.dtype:
            raise ValueError("k_pool / v_pool must both be bf16 or both fp32")
        if self.k_pool.dim() != 4 or self.v_pool.shape != self.k_pool.shape:
            raise ValueError("pools must be [num_pages, Hkv, page_size, D] and equal in shape")
        _need(self.k_pool, "k_pool")
        _need(self.v_pool, "v_pool")
        _need(self.page_table, "page_table", torch.int32)
        _need(self.ctx_len, "ctx_len", torch.int32)
        if self.page_table.dim() != 2 or self.ctx_len.dim() != 1 or \
                self.ctx_len.shape[0] != self.page_table.shape[0]:
            raise ValueError("page_table must be [B, max_pages] and ctx_len [B]")

    @property
    def dtype(self) -> torch.dtype:
        return self.k_pool.dtype

    @property
    def n_kv_heads(self) -> int:
        return int(self.k_pool.shape[1])

    @property
    def page_size(self) -> int:
        return int(self.k_pool.shape[2])

    @property
    def head_dim(self) -> int:
        return int(self.k_pool.shape[3])

    def struct(self) -> N.tt_kv_cache:
        c = N.tt_kv_cache()
        c.k_pool = self.k_pool.data_ptr()
        c.v_pool = self.v_pool.data_ptr()
        c.page_table = self.page_table.data_ptr()
        c.ctx_len = self.ctx_len.data_ptr()
        c.num_pages = int(self.k_pool.shape[0])
        c.max_pages_per_seq = int(self.page_table.shape[1])
        c.page_size = self.page_size
        c.n_kv_heads = self.n_kv_heads
        c.head_dim = self.head_dim
        c.dtype = _DT[self.dtype]
        return c


# ----------------------------------------------------------------------------- workspace

def tt_denoise_attn_workspace_size(B: int, S: int, Hq: int, Hkv: int, D: int, dtype: torch.dtype) -> int:
    n = ctypes.c_size_t(0)
    N.check(N.lib().tt_denoise_attn_workspace_size(B, S, Hq, Hkv, D, _DT[dtype], ctypes.byref(n)),
            "tt_denoise_attn_workspace_size")
    return int(n.value)


def tt_unmask_workspace_size(B: int, S: int, V: int, dtype: torch.dtype) -> int:
    n = ctypes.c_size_t(0)
    N.check(N.lib().tt_unmask_workspace_size(B, S, V, _DT[dtype], ctypes.byref(n)), "tt_unmask_workspace_size")
    return int(n.value)


def tt_block_step_workspace_size(B: int, S: int, Hq: int, Hkv: int, D: int, V: int, dtype: torch.dtype) -> int:
    n = ctypes.c_size_t(0)
    N.check(N.lib().tt_block_step_workspace_size(B, S, Hq, Hkv, D, V, _DT[dtype], ctypes.byref(n)),
            "tt_block_step_workspace_size")
    return int(n.value)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace buffer (the library requires zeros before first use)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def error_word(device="cuda") -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device)


# ----------------------------------------------------------------------------- calls

def tt_denoise_attn(cache: KVCache, q: torch.Tensor, k_blk: torch.Tensor, v_blk: torch.Tensor,
                    out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                    sm_scale: Optional[float] = None, max_ctas: int = 0,
                    ws: Optional[torch.Tensor] = None, dev_err: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Two-segment attention of one layer; q [B,S,Hq,D], k_blk/v_blk [B,S,Hkv,D] -> out [B,S,Hq,D]."""
    return _attention("tt_denoise_attn", cache, q, k_blk, v_blk, out, lse, sm_scale, max_ctas, ws, dev_err,
                      stream)


def tt_context_block_attn(cache: KVCache, q: torch.Tensor, k_blk: torch.Tensor, v_blk: torch.Tensor,
                          out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                          sm_scale: Optional[float] = None, max_ctas: int = 0,
                          ws: Optional[torch.Tensor] = None, dev_err: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """The context tower's attention over a committed block: as tt_denoise_attn, but block
    query i sees block keys 0..i only."""
    return _attention("tt_context_block_attn", cache, q, k_blk, v_blk, out, lse, sm_scale, max_ctas, ws,
                      dev_err, stream)


def _attention(name, cache, q, k_blk, v_blk, out, lse, sm_scale, max_ctas, ws, dev_err, stream):
    B, S, Hq, D = q.shape
    Hkv = cache.n_kv_heads
    _cover(cache, B)
    _need(q, "q", cache.dtype)
    _need(k_blk, "k_blk", cache.dtype, (B, S, Hkv, D))
    _need(v_blk, "v_blk", cache.dtype, (B, S, Hkv, D))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", cache.dtype, q.shape)
    _need(lse, "lse", torch.float32, (B, Hq, S), allow_none=True)
    err = _err(dev_err)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if ws is None:
        ws = workspace(tt_denoise_attn_workspace_size(B, S, Hq, Hkv, D, cache.dtype), q.device)
    wp, wb = _ws(ws)
    st = cache.struct()
    N.check(getattr(N.lib(), name)(ctypes.byref(st), q.data_ptr(), k_blk.data_ptr(), v_blk.data_ptr(),
                                   out.data_ptr(), _ptr(lse), B, S, Hq, float(sm_scale), int(max_ctas),
                                   wp, wb, err, _stream(stream)),
            name)
    return out


def tt_unmask(logits: torch.Tensor, masked: torch.Tensor, tokens: torch.Tensor, tau: float, step: int, T: int,
              committed_now: Optional[torch.Tensor] = None, conf: Optional[torch.Tensor] = None,
              n_masked: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
              dev_err: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Confidence unmasking in place: logits [B,S,V]; masked [B,S] uint8; tokens [B,S] int32."""
    B, S, V = logits.shape
    if logits.dtype not in _DT:
        raise ValueError("logits must be bf16 or fp32")
    _need(logits, "logits")
    _need(masked, "masked", torch.uint8, (B, S))
    _need(tokens, "tokens", torch.int32, (B, S))
    _need(committed_now, "committed_now", torch.uint8, (B, S), allow_none=True)
    _need(conf, "conf", torch.float32, (B, S), allow_none=True)
    _need(n_masked, "n_masked", torch.int32, (B,), allow_none=True)
    err = _err(dev_err)
    if ws is None:
        ws = workspace(tt_unmask_workspace_size(B, S, V, logits.dtype), logits.device)
    wp, wb = _ws(ws)
    N.check(N.lib().tt_unmask(logits.data_ptr(), _DT[logits.dtype], B, S, V, float(tau), int(step), int(T),
                              masked.data_ptr(), tokens.data_ptr(), _ptr(committed_now), _ptr(conf),
                              _ptr(n_masked), wp, wb, err, _stream(stream)),
            "tt_unmask")


def tt_unmask_noalloc(logits: torch.Tensor, masked: torch.Tensor, tokens: torch.Tensor, tau: float, step: int,
                      T: int, committed_now: Optional[torch.Tensor] = None, conf: Optional[torch.Tensor] = None,
                      n_masked: Optional[torch.Tensor] = None, dev_err: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> None:
    """tt_unmask without a workspace, for callers that cannot allocate device memory (inside
    graph capture, under a framework that owns the device pool, fixed-memory loops).  The
    library's own file-scope scratch array is used instead; every call shares it, so calls
    must not overlap on the GPU.  Make the first call on a device outside stream capture."""
    B, S, V = logits.shape
    if logits.dtype not in _DT:
        raise ValueError("logits must be bf16 or fp32")
    _need(logits, "logits")
    _need(masked, "masked", torch.uint8, (B, S))
    _need(tokens, "tokens", torch.int32, (B, S))
    _need(committed_now, "committed_now", torch.uint8, (B, S), allow_none=True)
    _need(conf, "conf", torch.float32, (B, S), allow_none=True)
    _need(n_masked, "n_masked", torch.int32, (B,), allow_none=True)
    err = _err(dev_err)
    N.check(N.lib().tt_unmask_noalloc(logits.data_ptr(), _DT[logits.dtype], B, S, V, float(tau), int(step),
                                      int(T), masked.data_ptr(), tokens.data_ptr(), _ptr(committed_now),
                                      _ptr(conf), _ptr(n_masked), err, _stream(stream)),
            "tt_unmask_noalloc")


def tt_linear_schedule_mask(u: torch.Tensor, t: torch.Tensor, masked: Optional[torch.Tensor] = None,
                            clean: Optional[torch.Tensor] = None, mask_id: int = -1,
                            noisy: Optional[torch.Tensor] = None, dev_err: Optional[torch.Tensor] = None,
                            stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Linear-schedule corruption: masked[b,p] = u[b,p] < t[b]; with ``noisy`` (and ``clean``)
    also noisy = mask_id where masked, clean elsewhere.  u [B,S] fp32, t [B] fp32."""
    B, S = u.shape
    _need(u, "u", torch.float32, (B, S))
    _need(t, "t", torch.float32, (B,))
    if masked is None:
        masked = torch.empty((B, S), dtype=torch.uint8, device=u.device)
    _need(masked, "masked", torch.uint8, (B, S))
    _need(clean, "clean", torch.int32, (B, S), allow_none=True)
    _need(noisy, "noisy", torch.int32, (B, S), allow_none=True)
    err = _err(dev_err)
    N.check(N.lib().tt_linear_schedule_mask(_ptr(clean), u.data_ptr(), t.data_ptr(), B, S, int(mask_id),
                                            _ptr(noisy), masked.data_ptr(), err, _stream(stream)),
            "tt_linear_schedule_mask")
    return masked


def tt_masked_nll_workspace_size(B: int, S: int, V: int, dtype: torch.dtype) -> int:
    n = ctypes.c_size_t(0)
    N.check(N.lib().tt_masked_nll_workspace_size(B, S, V, _DT[dtype], ctypes.byref(n)),
            "tt_masked_nll_workspace_size")
    return int(n.value)


def tt_masked_nll(logits: torch.Tensor, targets: torch.Tensor, masked: torch.Tensor,
                  nll: Optional[torch.Tensor] = None, nll_sum: Optional[torch.Tensor] = None,
                  count: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None,
                  dev_err: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None):
    """Masked-diffusion loss: logits [B,S,V]; targets [B,S] int32; masked [B,S] uint8.
    Returns (nll [B,S] fp32, NaN where unmasked; nll_sum [B] fp32; count [B] int32)."""
    B, S, V = logits.shape
    if logits.dtype not in _DT:
        raise ValueError("logits must be bf16 or fp32")
    _need(logits, "logits")
    _need(targets, "targets", torch.int32, (B, S))
    _need(masked, "masked", torch.uint8, (B, S))
    dev = logits.device
    if nll is None:
        nll = torch.empty((B, S), dtype=torch.float32, device=dev)
    if nll_sum is None:
        nll_sum = torch.empty((B,), dtype=torch.float32, device=dev)
    if count is None:
        count = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(nll, "nll", torch.float32, (B, S))
    _need(nll_sum, "nll_sum", torch.float32, (B,))
    _need(count, "count", torch.int32, (B,))
    err = _err(dev_err)
    if ws is None:
        ws = workspace(tt_masked_nll_workspace_size(B, S, V, logits.dtype), dev)
    wp, wb = _ws(ws)
    N.check(N.lib().tt_masked_nll(logits.data_ptr(), _DT[logits.dtype], B, S, V, targets.data_ptr(),
                                  masked.data_ptr(), nll.data_ptr(), nll_sum.data_ptr(), count.data_ptr(),
                                  wp, wb, err, _stream(stream)),
            "tt_masked_nll")
    return nll, nll_sum, count


def tt_kv_append(caches: Sequence[KVCache], k_new: Sequence[torch.Tensor], v_new: Sequence[torch.Tensor],
                 seq_active: Optional[torch.Tensor] = None, dev_err: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None) -> None:
    """Append one block per layer (k_new[l], v_new[l]: [B,S,Hkv,D]) and advance the shared ctx_len once."""
    n = len(caches)
    if n == 0 or len(k_new) != n or len(v_new) != n:
        raise ValueError("one k_new / v_new per cache")
    B, S = k_new[0].shape[:2]
    for l in range(n):
        shp = (B, S, caches[l].n_kv_heads, caches[l].head_dim)
        _need(k_new[l], f"k_new[{l}]", caches[l].dtype, shp)
        _need(v_new[l], f"v_new[{l}]", caches[l].dtype, shp)
    _need(seq_active, "seq_active", torch.uint8, (B,), allow_none=True)
    for c in caches:
        _cover(c, B)
    err = _err(dev_err)
    structs = (N.tt_kv_cache * n)(*[c.struct() for c in caches])
    N.check(N.lib().tt_kv_append(structs, n, N.ptr_array([t.data_ptr() for t in k_new]),
                                 N.ptr_array([t.data_ptr() for t in v_new]), _ptr(seq_active), B, S,
                                 err, _stream(stream)),
            "tt_kv_append")


def tt_block_step(caches: Sequence[KVCache], q: Sequence[torch.Tensor], k_blk: Sequence[torch.Tensor],
                  v_blk: Sequence[torch.Tensor], out: Sequence[torch.Tensor], logits: torch.Tensor,
                  masked: torch.Tensor, tokens: torch.Tensor, tau: float, step: int, T: int,
                  sm_scale: Optional[float] = None, committed_now: Optional[torch.Tensor] = None,
                  conf: Optional[torch.Tensor] = None, n_masked: Optional[torch.Tensor] = None,
                  ws: Optional[torch.Tensor] = None, dev_err: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None) -> None:
    """One denoiser step: attention for every layer, then unmasking of the step's logits."""
    n = len(caches)
    if not (len(q) == len(k_blk) == len(v_blk) == len(out) == n) or n == 0:
        raise ValueError("one q / k_blk / v_blk / out per layer")
    B, S, Hq, D = q[0].shape
    V = logits.shape[2]
    dt = caches[0].dtype
    for l in range(n):
        _cover(caches[l], B)
        _need(q[l], f"q[{l}]", dt, (B, S, Hq, D))
        _need(k_blk[l], f"k_blk[{l}]", dt, (B, S, caches[l].n_kv_heads, D))
        _need(v_blk[l], f"v_blk[{l}]", dt, (B, S, caches[l].n_kv_heads, D))
        _need(out[l], f"out[{l}]", dt, (B, S, Hq, D))
    _need(logits, "logits", dt, (B, S, V))
    _need(masked, "masked", torch.uint8, (B, S))
    _need(tokens, "tokens", torch.int32, (B, S))
    _need(committed_now, "committed_now", torch.uint8, (B, S), allow_none=True)
    _need(conf, "conf", torch.float32, (B, S), allow_none=True)
    _need(n_masked, "n_masked", torch.int32, (B,), allow_none=True)
    err = _err(dev_err)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if ws is None:
        ws = workspace(tt_block_step_workspace_size(B, S, Hq, caches[0].n_kv_heads, D, V, dt), logits.device)
    wp, wb = _ws(ws)
    structs = (N.tt_kv_cache * n)(*[c.struct() for c in caches])
    N.check(N.lib().tt_block_step(structs, n, N.ptr_array([t.data_ptr() for t in q]),
                                  N.ptr_array([t.data_ptr() for t in k_blk]),
                                  N.ptr_array([t.data_ptr() for t in v_blk]),
                                  N.ptr_array([t.data_ptr() for t in out]), logits.data_ptr(), B, S, Hq, V,
                                  float(tau), int(step), int(T), float(sm_scale), masked.data_ptr(),
                                  tokens.data_ptr(), _ptr(committed_now), _ptr(conf), _ptr(n_masked),
                                  wp, wb, err, _stream(stream)),
            "tt_block_step")


def tt_get_device_error(dev_err: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise the stream and return the device error word (0 = no error)."""
    code = ctypes.c_uint32(0)
    _need(dev_err, "dev_err", torch.int32)
    N.check(N.lib().tt_get_device_error(dev_err.data_ptr(), _stream(stream), ctypes.byref(code)),
            "tt_get_device_error")
    return int(code.value)


def tt_check_wait_timeout(polls: int, dev_err: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Launch the library's bounded-wait self-check: a wait that can never finish gives up
    after `polls` polls and records TT_ERR_DEVICE_TIMEOUT in `dev_err` (read it with
    tt_get_device_error)."""
    _need(dev_err, "dev_err", dtype=torch.int32)
    N.check(N.lib().tt_check_wait_timeout(int(polls), dev_err.data_ptr(), _stream(stream)), "tt_check_wait_timeout")
