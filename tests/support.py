"""Helpers of the GPU parity tests: move seeded inputs to the device and compare the
CUDA path's results with the float64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from block_wise_diffusion_denoise_b300 import synth
from block_wise_diffusion_denoise_b300.api import KVCache

TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}
NEAR_TAU = 1e-4          # positions whose oracle confidence is this close to tau are not compared
FALLBACK_TIE = 1e-5      # relative gap under which two confidences count as tied for the fallback


def to_dev(arr: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).cuda()


def to_host_bits(t: torch.Tensor, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.detach().cpu().numpy()


def to_host_f64(t: torch.Tensor, dtype: str) -> np.ndarray:
    return oracle.decode(to_host_bits(t, dtype), dtype)


def cache_to_dev(c: synth.PagedCache) -> KVCache:
    return KVCache(to_dev(c.k_pool, c.dtype), to_dev(c.v_pool, c.dtype),
                   torch.from_numpy(c.page_table.astype(np.int32)).cuda(),
                   torch.from_numpy(c.ctx_len.astype(np.int32)).cuda())


def attention_case(cfg: synth.StepConfig, seed=0, lens=None, capacity=None, garbage=None, layer=0,
                   block=0, step=0):
    """Seeded inputs of one attention layer: (host cache, q, k_blk, v_blk)."""
    lens = synth.draw_lengths(cfg, seed) if lens is None else np.asarray(lens, np.int32)
    cap = int(max(lens.max(), 1) + cfg.S) if capacity is None else capacity
    cache = synth.draw_paged_cache(cfg, lens, cap, seed=seed, layer=layer, garbage=garbage)
    q, kb, vb = synth.draw_block_qkv(cfg, seed=seed, block=block, step=step, layer=layer)
    return cache, q, kb, vb


def oracle_attention(cfg, cache, q, kb, vb, sm_scale, seqs=None):
    return oracle.denoise_attention(cache.k_pool, cache.v_pool, cache.page_table, cache.ctx_len,
                                    cache.page_size, q, kb, vb, sm_scale, cfg.dtype, seqs=seqs)


def max_abs(a, b):
    return float(np.nanmax(np.abs(a - b))) if a.size else 0.0


def compare_unmask(pre_masked, pre_tokens, ora, gpu_masked, gpu_tokens, gpu_committed, gpu_conf,
                   gpu_nmasked, tau, step, T):
    """Bit-exact comparison of one unmasking step, sequence by sequence.

    A position whose oracle confidence lies within NEAR_TAU of tau is excluded; if
    such a position could decide whether the commit set is empty (every other masked
    position is below tau), the whole sequence is excluded, and so is a sequence whose
    fallback choice is a near tie.  Committed tokens are always compared (the argmax
    is exact on both sides).  A sequence whose oracle entry is None (not sampled) gets the
    checks that need no oracle: only masked positions commit, locked ones never change, at
    least one position commits while any is masked, everything commits at step T, and the
    count of positions left matches the mask.  Returns (excluded positions, excluded sequences)."""
    B, S = pre_masked.shape
    ex_pos = ex_seq = 0
    for b in range(B):
        r = ora[b]
        m0 = pre_masked[b].astype(bool)
        if r is None:
            com = gpu_committed[b].astype(bool)
            assert not (com & ~m0).any(), (b, "committed a locked position")
            assert np.array_equal(gpu_tokens[b][~m0], pre_tokens[b][~m0])
            assert np.array_equal(gpu_masked[b].astype(bool), m0 & ~com), b
            assert (gpu_tokens[b][com] >= 0).all()
            assert np.isnan(gpu_conf[b][~m0]).all() and np.isfinite(gpu_conf[b][m0]).all()
            if m0.any():
                assert com.any(), (b, "nothing committed")
            if step >= T:
                assert np.array_equal(com, m0)
            assert gpu_nmasked[b] == int(gpu_masked[b].sum())
            continue
        # the argmax of every committed position is exact on both sides
        for p in np.nonzero(gpu_committed[b])[0]:
            assert m0[p], (b, p, "committed a locked position")
            assert gpu_tokens[b, p] == r.argmax[p], (b, p, gpu_tokens[b, p], r.argmax[p])
        # locked positions never change
        assert np.array_equal(gpu_tokens[b][~m0], pre_tokens[b][~m0])
        assert not gpu_masked[b][~m0].any()
        # confidence (fp32 on the device)
        if m0.any():
            rel = np.abs(gpu_conf[b][m0] - r.conf[m0]) / r.conf[m0]
            assert rel.max() < 1e-5, (b, rel.max())
        assert np.isnan(gpu_conf[b][~m0]).all()
        if step >= T:
            assert np.array_equal(gpu_committed[b].astype(bool), m0)
            assert not gpu_masked[b].any() and gpu_nmasked[b] == 0
            continue
        near = m0 & (np.abs(np.nan_to_num(r.conf, nan=-1.0) - tau) < NEAR_TAU)
        clear_above = m0 & ~near & (np.nan_to_num(r.conf, nan=-1.0) >= tau)
        excluded = False
        if near.any() and not clear_above.any():
            excluded = True
        if r.fallback and not near.any():
            c = np.sort(r.conf[m0])[::-1]
            if c.size > 1 and (c[0] - c[1]) <= FALLBACK_TIE * c[0]:
                excluded = True
        if excluded:
            ex_seq += 1
            ex_pos += int(near.sum())
            assert gpu_committed[b].sum() >= 1 if m0.any() else True
            continue
        ex_pos += int(near.sum())
        keep = ~near
        assert np.array_equal(gpu_committed[b][keep].astype(bool), r.committed_now[keep]), b
        assert np.array_equal(gpu_masked[b][keep].astype(bool), r.masked[keep]), b
        assert np.array_equal(gpu_tokens[b][keep], r.tokens[keep]), b
        if not near.any():
            assert gpu_nmasked[b] == int(r.masked.sum())
    return ex_pos, ex_seq
