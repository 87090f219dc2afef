"""Two-segment denoise attention on the GPU (tt_denoise_attn) against the float64 oracle.

Tolerances: max-abs 1e-5 in fp32 mode, 2e-2 in bf16.  Because the seeded workload
(Q, K ~ N(0,1)/sqrt(D) with a further 1/sqrt(D) softmax scale) gives nearly uniform
attention, the bf16 cases also run a stress variant with unscaled N(0,1) inputs and
keys planted to dominate at page and split edges, where a dropped or misplaced key
shows up far above the tolerance."""
import math

import numpy as np
import pytest
import torch

import oracle
from block_wise_diffusion_denoise_b300 import _native as N
from block_wise_diffusion_denoise_b300 import api, synth
from tests import support

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}


def _run(cfg, cache_h, q, kb, vb, max_ctas=0, ws=None, check_err=True, scale=None):
    cache = support.cache_to_dev(cache_h)
    qd, kd, vd = (support.to_dev(x, cfg.dtype) for x in (q, kb, vb))
    lse = torch.full((cfg.B, cfg.Hq, cfg.S), float("nan"), device="cuda")
    err = api.error_word()
    scale = 1.0 / math.sqrt(cfg.D) if scale is None else scale
    out = api.tt_denoise_attn(cache, qd, kd, vd, lse=lse, sm_scale=scale, max_ctas=max_ctas, ws=ws, dev_err=err)
    code = api.tt_get_device_error(err)
    if check_err:
        assert code == 0, code
    return support.to_host_f64(out, cfg.dtype), lse.cpu().numpy().astype(np.float64), code, out


def _oracle_groups(cfg, cache_h, q, kb, vb, pairs, scale=None):
    """Oracle output of selected (sequence, KV head) pairs: dict (b, g) -> (o [S,G,D], lse [G,S])."""
    scale = 1.0 / math.sqrt(cfg.D) if scale is None else scale
    res = {}
    for b, g in pairs:
        L = int(cache_h.ctx_len[b])
        kc = oracle.decode(oracle.context_rows(cache_h.k_pool, cache_h.page_table[b], L, cfg.page_size), cfg.dtype)
        vc = oracle.decode(oracle.context_rows(cache_h.v_pool, cache_h.page_table[b], L, cfg.page_size), cfg.dtype)
        hs = slice(g * cfg.G, (g + 1) * cfg.G)
        res[(b, g)] = oracle.denoise_attention_seq(
            oracle.decode(q[b][:, hs], cfg.dtype), kc[:, g:g + 1], vc[:, g:g + 1],
            oracle.decode(kb[b][:, g:g + 1], cfg.dtype), oracle.decode(vb[b][:, g:g + 1], cfg.dtype),
            scale)
    return res


def _check(cfg, cache_h, q, kb, vb, pairs=None, max_ctas=0, tol=None, scale=None):
    o, lse, _, _ = _run(cfg, cache_h, q, kb, vb, max_ctas=max_ctas, scale=scale)
    if pairs is None:
        pairs = [(b, g) for b in range(cfg.B) for g in range(cfg.Hkv)]
    want = _oracle_groups(cfg, cache_h, q, kb, vb, pairs, scale=scale)
    tol = TOL[cfg.dtype] if tol is None else tol
    worst = 0.0
    for (b, g), (wo, wl) in want.items():
        hs = slice(g * cfg.G, (g + 1) * cfg.G)
        err = support.max_abs(o[b][:, hs], wo)
        worst = max(worst, err)
        assert err <= tol, ((b, g), err)
        assert support.max_abs(lse[b][hs], wl) <= max(1e-4, tol), ((b, g), support.max_abs(lse[b][hs], wl))
    return o, worst


# ----------------------------------------------------------------------------- fp32 mode

def test_tiny_fp32():
    cfg = synth.CONFIGS["tiny"]
    _check(cfg, *support.attention_case(cfg, seed=0))


@pytest.mark.parametrize("L", [0, 1, 15, 37, 64, 65, 200])
def test_fp32_context_lengths(L):
    cfg = synth.CONFIGS["tiny"].replace(B=2, qkv_scale=1.0)
    _check(cfg, *support.attention_case(cfg, seed=L, lens=[L, max(0, L - 3)]))


def test_fp32_block_only_matches_plain_bidirectional_attention():
    """L = 0: the result is ordinary softmax attention inside the block."""
    cfg = synth.CONFIGS["tiny"].replace(B=1, qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=4, lens=[0])
    o, _, _, _ = _run(cfg, cache, q, kb, vb)
    qq, kk, vv = (oracle.decode(x[0], "f32") for x in (q, kb, vb))
    for h in range(cfg.Hq):
        s = qq[:, h] @ kk[:, h // cfg.G].T / math.sqrt(cfg.D)
        p = np.exp(s - s.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        assert np.abs(o[0][:, h] - p @ vv[:, h // cfg.G]).max() < 1e-5


# ----------------------------------------------------------------------------- bf16

def test_single_bf16_full():
    cfg = synth.CONFIGS["single"]
    _check(cfg, *support.attention_case(cfg, seed=0))


def test_single_bf16_stress_planted_keys():
    cfg = synth.CONFIGS["single"].replace(qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=1)
    synth.plant_keys(cfg, cache, q, seed=1, per_seq=12, boost=0.5)
    o, worst = _check(cfg, cache, q, kb, vb)


@pytest.mark.parametrize("lens", [[0, 1, 63, 64], [65, 127, 129, 1000], [4095, 4097, 16, 5000]])
def test_bf16_ragged_edges(lens):
    cfg = synth.CONFIGS["ragged"].replace(B=len(lens), qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=sum(lens), lens=lens)
    synth.plant_keys(cfg, cache, q, seed=2, per_seq=6, boost=0.5)
    _check(cfg, cache, q, kb, vb)


def test_ragged_config_sampled():
    """The ragged batch (B=32, L ~ U[1024, 8192]) at full size; the oracle checks sampled pairs."""
    cfg = synth.CONFIGS["ragged"]
    cache, q, kb, vb = support.attention_case(cfg, seed=0)
    lens = cache.ctx_len
    pairs = [(int(np.argmin(lens)), 0), (int(np.argmax(lens)), 1), (7, 0), (31, 1)]
    _check(cfg, cache, q, kb, vb, pairs=pairs)


def test_ctx8k_sampled_and_stress():
    cfg = synth.CONFIGS["ctx8k"]
    cache, q, kb, vb = support.attention_case(cfg, seed=0)
    _check(cfg, cache, q, kb, vb, pairs=[(0, 0), (13, 1), (31, 0)])
    cfg2 = cfg.replace(qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg2, seed=3)
    synth.plant_keys(cfg2, cache, q, seed=3, per_seq=8, boost=0.5)
    _check(cfg2, cache, q, kb, vb, pairs=[(2, 1), (17, 0), (30, 1)])


def test_long_context_sampled():
    cfg = synth.CONFIGS["long"].replace(qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=0)
    synth.plant_keys(cfg, cache, q, seed=4, per_seq=16, boost=0.5)
    _check(cfg, cache, q, kb, vb, pairs=[(1, 0), (3, 1)])


# ----------------------------------------------------------------------------- invariances

@pytest.mark.parametrize("name", ["tiny", "single"])
def test_garbage_in_unused_slots_changes_nothing(name):
    """NaN / huge values in page slots at or beyond L and in unowned pages: bitwise equal output."""
    cfg = synth.CONFIGS[name].replace(B=3)
    lens = np.array([cfg.len_lo, 37, 0], np.int32)
    base = support.attention_case(cfg, seed=5, lens=lens, capacity=int(lens.max()) + 200)
    o0 = _run(cfg, *base)[3]
    for kind in ("nan", "huge"):
        g = support.attention_case(cfg, seed=5, lens=lens, capacity=int(lens.max()) + 200, garbage=kind)
        o1 = _run(cfg, *g)[3]
        assert torch.equal(o0.view(torch.int16) if o0.dtype == torch.bfloat16 else o0,
                           o1.view(torch.int16) if o1.dtype == torch.bfloat16 else o1), kind


@pytest.mark.parametrize("name", ["tiny", "single"])
def test_physical_page_order_is_irrelevant(name):
    cfg = synth.CONFIGS[name].replace(B=2)
    cache, q, kb, vb = support.attention_case(cfg, seed=6, lens=[cfg.len_lo, cfg.len_lo // 2 + 3])
    o0 = _run(cfg, cache, q, kb, vb)[3]
    rng = np.random.default_rng(0)
    perm = rng.permutation(cache.num_pages)           # new physical slot of every page
    k2, v2 = np.empty_like(cache.k_pool), np.empty_like(cache.v_pool)
    k2[perm], v2[perm] = cache.k_pool, cache.v_pool
    moved = synth.PagedCache(k2, v2, perm[cache.page_table].astype(np.int32), cache.ctx_len.copy(),
                             cache.page_size, cache.dtype)
    o1 = _run(cfg, moved, q, kb, vb)[3]
    assert torch.equal(o0, o1)


def test_split_count_does_not_change_the_result():
    cfg = synth.CONFIGS["single"].replace(B=2, qkv_scale=1.0)
    case = support.attention_case(cfg, seed=8, lens=[4096, 777])
    o_auto = _run(cfg, *case)[0]
    for k in (1, 3, 64):
        o_k = _run(cfg, *case, max_ctas=k)[0]
        assert support.max_abs(o_auto, o_k) <= 1e-2


def test_device_errors_are_reported():
    cfg = synth.CONFIGS["tiny"].replace(B=2)
    cache, q, kb, vb = support.attention_case(cfg, seed=9, lens=[64, 64])
    bad = synth.PagedCache(cache.k_pool, cache.v_pool, cache.page_table.copy(), cache.ctx_len.copy(),
                           cache.page_size, cache.dtype)
    bad.page_table[1, 0] = cache.num_pages + 5                     # page id outside the pool
    assert _run(cfg, bad, q, kb, vb, check_err=False)[2] == N.TT_ERR_BOUNDS
    long = synth.PagedCache(cache.k_pool, cache.v_pool, cache.page_table, np.array([64, 10 ** 6], np.int32),
                            cache.page_size, cache.dtype)
    assert _run(cfg, long, q, kb, vb, check_err=False)[2] == N.TT_ERR_BOUNDS


def test_batch_above_one_launch_table():
    """More sequences than one launch's sequence table holds (1024): the batch runs as several
    launches; sequences on both sides of the cut and at the ends match the oracle."""
    cfg = synth.CONFIGS["single"].replace(B=1100, Hq=16, Hkv=1, len_lo=0, len_hi=300,
                                          qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=21)
    pairs = [(b, 0) for b in (0, 1, 511, 1022, 1023, 1024, 1025, 1099)]
    _check(cfg, cache, q, kb, vb, pairs=pairs)


@pytest.mark.parametrize("S,Hq,Hkv", [(32, 32, 2), (64, 16, 2), (48, 16, 2), (128, 4, 2), (16, 24, 1)])
def test_tensor_core_shapes_beyond_two_m_tiles(S, Hq, Hkv):
    """Block sizes and head groupings with 3 to 16 M tiles of 128 rows per segment (S = 32, 48,
    64, 128; 24 query heads per KV head) on the tensor-core kernel, ragged contexts, stress
    values, against the oracle."""
    cfg = synth.CONFIGS["single"].replace(B=3, S=S, Hq=Hq, Hkv=Hkv, qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=S + Hq, lens=[0, 700, 1500])
    _check(cfg, cache, q, kb, vb)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_single_query_decode_shape(dtype):
    """S = 1 (one query per head, the autoregressive decode shape) on the same paged cache:
    the CUDA-core kernel, ragged lengths including 0, against the oracle."""
    base = synth.CONFIGS["single"] if dtype == "bf16" else synth.CONFIGS["tiny"]
    cfg = base.replace(B=4, S=1, qkv_scale=1.0)
    lens = [0, 1, 777, 4096] if dtype == "bf16" else [0, 1, 37, 64]
    _check(cfg, *support.attention_case(cfg, seed=31, lens=lens))


@pytest.mark.parametrize("name,scale", [("single", 0.3), ("single", 0.02), ("tiny", 0.5), ("single", -0.05)])
def test_softmax_scale_argument(name, scale):
    """Scales other than 1/sqrt(D): sharper and flatter weights on the tensor-core kernel, the
    fp32 kernel, and a negative scale (taken by the CUDA-core kernel), with the LSE."""
    cfg = synth.CONFIGS[name].replace(B=2, qkv_scale=1.0)
    lens = [cfg.len_lo, 130] if name == "single" else [64, 5]
    _check(cfg, *support.attention_case(cfg, seed=33, lens=lens), scale=scale)
