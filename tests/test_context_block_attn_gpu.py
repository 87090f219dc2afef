"""The context tower's attention over a committed block (tt_context_block_attn) on the GPU
against the float64 oracle's causal-block view: block query i sees every context key and the
block keys 0..i.

Tolerances as for tt_denoise_attn: max-abs 1e-5 in fp32 mode, 2e-2 in bf16.  Short contexts
and block keys planted to dominate one (position, head) row make the block segment carry most
of the weight, so a key let through or held back by the mask shows far above the tolerance."""
import math

import numpy as np
import pytest
import torch

import oracle
from block_wise_diffusion_denoise_b300 import api, synth
from tests import support

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}


def _run(cfg, cache_h, q, kb, vb, causal=True, max_ctas=0):
    cache = support.cache_to_dev(cache_h)
    qd, kd, vd = (support.to_dev(x, cfg.dtype) for x in (q, kb, vb))
    lse = torch.full((cfg.B, cfg.Hq, cfg.S), float("nan"), device="cuda")
    err = api.error_word()
    fn = api.tt_context_block_attn if causal else api.tt_denoise_attn
    out = fn(cache, qd, kd, vd, lse=lse, sm_scale=1.0 / math.sqrt(cfg.D), max_ctas=max_ctas, dev_err=err)
    assert api.tt_get_device_error(err) == 0
    return support.to_host_f64(out, cfg.dtype), lse.cpu().numpy().astype(np.float64)


def _plant_block_keys(cfg, q, kb, seed, boost=0.5):
    """Per sequence and KV head, make two block keys dominate one query row each."""
    rng = np.random.default_rng(seed)
    for b in range(cfg.B):
        for g in range(cfg.Hkv):
            for j in rng.choice(cfg.S, size=min(2, cfg.S), replace=False):
                s = int(rng.integers(0, cfg.S))
                h = g * cfg.G + int(rng.integers(0, cfg.G))
                qv = (oracle.decode(q[b, s, h], cfg.dtype) * boost).astype(np.float32)
                kb[b, j, g] = synth.bf16_bits(qv) if cfg.dtype == "bf16" else qv


def _check(cfg, cache_h, q, kb, vb, pairs=None, max_ctas=0):
    o, lse = _run(cfg, cache_h, q, kb, vb, max_ctas=max_ctas)
    if pairs is None:
        pairs = [(b, g) for b in range(cfg.B) for g in range(cfg.Hkv)]
    tol = TOL[cfg.dtype]
    for b, g in pairs:
        L = int(cache_h.ctx_len[b])
        kc = oracle.decode(oracle.context_rows(cache_h.k_pool, cache_h.page_table[b], L, cfg.page_size), cfg.dtype)
        vc = oracle.decode(oracle.context_rows(cache_h.v_pool, cache_h.page_table[b], L, cfg.page_size), cfg.dtype)
        hs = slice(g * cfg.G, (g + 1) * cfg.G)
        wo, wl = oracle.denoise_attention_seq(
            oracle.decode(q[b][:, hs], cfg.dtype), kc[:, g:g + 1], vc[:, g:g + 1],
            oracle.decode(kb[b][:, g:g + 1], cfg.dtype), oracle.decode(vb[b][:, g:g + 1], cfg.dtype),
            1.0 / math.sqrt(cfg.D), causal_block=True)
        err = support.max_abs(o[b][:, hs], wo)
        assert err <= tol, ((b, g), err)
        assert support.max_abs(lse[b][hs], wl) <= max(1e-4, tol), ((b, g), support.max_abs(lse[b][hs], wl))
    return o


@pytest.mark.parametrize("L", [0, 1, 37, 65])
def test_fp32_context_lengths(L):
    cfg = synth.CONFIGS["tiny"].replace(B=2, qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=40 + L, lens=[L, max(0, L - 3)])
    _plant_block_keys(cfg, q, kb, seed=L)
    _check(cfg, cache, q, kb, vb)


def test_bf16_tensor_core_ragged_with_planted_block_keys():
    cfg = synth.CONFIGS["single"].replace(B=4, qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=41, lens=[0, 63, 130, 4096])
    _plant_block_keys(cfg, q, kb, seed=41)
    _check(cfg, cache, q, kb, vb)


@pytest.mark.parametrize("S,Hq,Hkv", [(32, 32, 2), (64, 16, 2), (128, 4, 2), (16, 24, 1)])
def test_tensor_core_shapes_beyond_two_m_tiles(S, Hq, Hkv):
    """Block rows r = s * G + h spread over 3 to 16 M tiles: each row's mask comes from its own
    block position."""
    cfg = synth.CONFIGS["single"].replace(B=3, S=S, Hq=Hq, Hkv=Hkv, qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=S + Hq + 1, lens=[0, 300, 1500])
    _plant_block_keys(cfg, q, kb, seed=S)
    _check(cfg, cache, q, kb, vb)


@pytest.mark.parametrize("max_ctas", [1, 3, 64])
def test_split_segments_merge_the_causal_block_tile(max_ctas):
    cfg = synth.CONFIGS["single"].replace(B=2, qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=42, lens=[4096, 777])
    _plant_block_keys(cfg, q, kb, seed=42)
    _check(cfg, cache, q, kb, vb, max_ctas=max_ctas)


def test_ctx8k_sampled():
    cfg = synth.CONFIGS["ctx8k"].replace(qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=43)
    _plant_block_keys(cfg, q, kb, seed=43, boost=1.0)
    _check(cfg, cache, q, kb, vb, pairs=[(0, 1), (19, 0), (31, 1)])


@pytest.mark.parametrize("name", ["tiny", "single"])
def test_last_position_matches_the_denoiser_view_and_earlier_ones_do_not(name):
    """The last block position sees every key in both views; with no context, every earlier
    position sees fewer keys and its output moves."""
    cfg = synth.CONFIGS[name].replace(B=2, qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=44, lens=[0, 0])
    oc, lc = _run(cfg, cache, q, kb, vb, causal=True)
    ob, lb = _run(cfg, cache, q, kb, vb, causal=False)
    assert support.max_abs(oc[:, -1], ob[:, -1]) <= 1e-6
    assert support.max_abs(lc[:, :, -1], lb[:, :, -1]) <= 1e-6
    assert (np.abs(oc[:, :-1] - ob[:, :-1]).max(axis=(0, 2, 3)) > 0.05).all()
