"""Single-position attention (S = 1, 16 query heads per KV head, bf16, D = 128) on the GPU
against the float64 oracle.

A block of one token is one step of autoregressive decoding from the same paged cache:
the library serves it with its own tensor-core kernel (the 16 query heads of a KV head
share every K and V read).  Same tolerance as the block kernel: max-abs 2e-2 in bf16,
lse within 2e-2.  Most cases use unscaled N(0,1) inputs with keys planted at page,
tile and split edges, so that a dropped or misplaced key shows far above the tolerance."""
import numpy as np
import pytest
import torch

from block_wise_diffusion_denoise_b300 import _native as N
from block_wise_diffusion_denoise_b300 import api, synth
from tests import support
from tests.test_attn_gpu import _check, _run

pytestmark = pytest.mark.gpu


def _cfg(name, **kw):
    return synth.CONFIGS[name].replace(S=1, **kw)


@pytest.mark.parametrize("lens", [[0, 1, 15, 63], [64, 65, 127, 128], [129, 191, 192, 255],
                                  [1000, 4095, 4097, 16]])
def test_context_lengths_around_page_and_tile_edges(lens):
    cfg = _cfg("ragged", B=len(lens), qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=100 + sum(lens), lens=lens)
    synth.plant_keys(cfg, cache, q, seed=3, per_seq=6, boost=0.5)
    _check(cfg, cache, q, kb, vb)


def test_single_sequence_default_scale():
    cfg = _cfg("single")
    _check(cfg, *support.attention_case(cfg, seed=0))


def test_ragged_config_full_batch():
    """The ragged batch (B=32, L ~ U[1024, 8192]) with one position: every segment checked."""
    cfg = _cfg("ragged", qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=0)
    synth.plant_keys(cfg, cache, q, seed=5, per_seq=8, boost=0.5)
    _check(cfg, cache, q, kb, vb)


def test_ctx8k_sampled():
    cfg = _cfg("ctx8k", qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=1)
    synth.plant_keys(cfg, cache, q, seed=1, per_seq=8, boost=0.5)
    _check(cfg, cache, q, kb, vb, pairs=[(0, 0), (9, 1), (22, 0), (31, 1)])


def test_long_context_split_over_many_ctas():
    """B=4 x 131072: every segment is cut into stream-K pieces merged through partials."""
    cfg = _cfg("long", qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=2)
    synth.plant_keys(cfg, cache, q, seed=2, per_seq=16, boost=0.5)
    _check(cfg, cache, q, kb, vb, pairs=[(0, 1), (2, 0), (3, 1)])


def test_split_count_does_not_change_the_result():
    cfg = _cfg("single", B=3, qkv_scale=1.0)
    case = support.attention_case(cfg, seed=8, lens=[4096, 777, 0])
    o_auto = _run(cfg, *case)[0]
    for k in (1, 2, 3, 7, 64, 296):
        o_k = _run(cfg, *case, max_ctas=k)[0]
        assert support.max_abs(o_auto, o_k) <= 1e-2, k
    _check(cfg, *case, max_ctas=5)


def test_garbage_in_unused_slots_changes_nothing():
    """NaN / huge values in page slots at or beyond L and in unowned pages: bitwise equal output."""
    cfg = _cfg("single", B=3)
    lens = np.array([300, 37, 0], np.int32)
    base = support.attention_case(cfg, seed=5, lens=lens, capacity=int(lens.max()) + 200)
    o0 = _run(cfg, *base)[3]
    for kind in ("nan", "huge"):
        g = support.attention_case(cfg, seed=5, lens=lens, capacity=int(lens.max()) + 200, garbage=kind)
        o1 = _run(cfg, *g)[3]
        assert torch.equal(o0.view(torch.int16), o1.view(torch.int16)), kind


def test_context_block_view_is_the_same_for_one_position():
    """With one block position the causal view inside the block is the plain one."""
    cfg = _cfg("single", B=2, qkv_scale=1.0)
    cache_h, q, kb, vb = support.attention_case(cfg, seed=11, lens=[500, 2000])
    cache = support.cache_to_dev(cache_h)
    qd, kd, vd = (support.to_dev(x, cfg.dtype) for x in (q, kb, vb))
    a = api.tt_denoise_attn(cache, qd, kd, vd)
    b = api.tt_context_block_attn(cache, qd, kd, vd)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_batch_above_one_launch_table():
    cfg = _cfg("single", B=1100, Hq=16, Hkv=1, len_lo=0, len_hi=300, qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=21)
    _check(cfg, cache, q, kb, vb, pairs=[(0, 0), (1023, 0), (1024, 0), (1099, 0)])


def test_device_errors_are_reported():
    cfg = _cfg("single", B=2, qkv_scale=1.0)
    cache, q, kb, vb = support.attention_case(cfg, seed=9, lens=[64, 64])
    bad = synth.PagedCache(cache.k_pool, cache.v_pool, cache.page_table.copy(), cache.ctx_len.copy(),
                           cache.page_size, cache.dtype)
    bad.page_table[1, 0] = cache.num_pages + 5                     # page id outside the pool
    assert _run(cfg, bad, q, kb, vb, check_err=False)[2] == N.TT_ERR_BOUNDS
    long = synth.PagedCache(cache.k_pool, cache.v_pool, cache.page_table, np.array([64, 10 ** 6], np.int32),
                            cache.page_size, cache.dtype)
    assert _run(cfg, long, q, kb, vb, check_err=False)[2] == N.TT_ERR_BOUNDS


def test_repeated_calls_share_one_workspace():
    """Split launches leave the tickets as they found them: the same workspace serves every call."""
    cfg = _cfg("long", B=2, len_lo=20000, len_hi=20000, qkv_scale=1.0)
    case = support.attention_case(cfg, seed=12)
    ws = api.workspace(api.tt_denoise_attn_workspace_size(cfg.B, 1, cfg.Hq, cfg.Hkv, cfg.D, torch.bfloat16))
    first = _run(cfg, *case, ws=ws)[3]
    for _ in range(3):
        assert torch.equal(_run(cfg, *case, ws=ws)[3].view(torch.int16), first.view(torch.int16))
    assert int(ws[:256].view(torch.int32).abs().sum()) == 0


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("single", {"Hq": 16, "Hkv": 2}),
                                     ("single", {"Hq": 64, "Hkv": 2})])
def test_one_position_on_the_cuda_core_kernel(name, kw):
    """S = 1 shapes the decode kernel does not take (fp32; 8 or 32 query heads per KV head)
    run on the CUDA-core kernel, against the same oracle."""
    cfg = _cfg(name, B=3, qkv_scale=1.0, **kw)
    lens = [cfg.len_lo, 1, 0] if name == "tiny" else [700, 129, 0]
    cache, q, kb, vb = support.attention_case(cfg, seed=31, lens=lens)
    tol = 1e-5 if cfg.dtype == "f32" else 2e-2
    _check(cfg, cache, q, kb, vb, tol=tol)
