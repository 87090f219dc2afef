"""Block commit on the GPU (tt_kv_append) against the oracle's append: pages hold bitwise
copies of the new rows, lengths advance once, inactive sequences and foreign slots stay
untouched, and attention over the grown context matches the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from block_wise_diffusion_denoise_b300 import _native as N
from block_wise_diffusion_denoise_b300 import api, synth
from tests import support

pytestmark = pytest.mark.gpu


def _layers(cfg, lens, capacity, n_layers, seed=0):
    return [synth.draw_paged_cache(cfg, lens, capacity, seed=seed, layer=l) for l in range(n_layers)]


def _append(cfg, caches_h, k_new, v_new, active=None):
    devs = [support.cache_to_dev(c) for c in caches_h]
    shared = devs[0].ctx_len
    for d in devs:
        d.ctx_len = shared                     # the layers hold the same tokens: one length array
    err = api.error_word()
    act = None if active is None else torch.from_numpy(active.astype(np.uint8)).cuda()
    api.tt_kv_append(devs, [support.to_dev(k, cfg.dtype) for k in k_new],
                     [support.to_dev(v, cfg.dtype) for v in v_new], seq_active=act, dev_err=err)
    code = api.tt_get_device_error(err)
    return devs, code


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_append_matches_oracle_bitwise(dtype):
    cfg = synth.CONFIGS["loop"].replace(B=5, dtype=dtype, n_layers=3)
    lens = np.array([0, 50, 64, 100, 127], np.int32)        # straddles, starts and ends on page edges
    caches = _layers(cfg, lens, 256, cfg.n_layers)
    kn, vn = zip(*[synth.draw_new_block_kv(cfg, block=1, layer=l) for l in range(cfg.n_layers)])
    active = np.array([1, 1, 0, 1, 1], np.uint8)
    devs, code = _append(cfg, caches, kn, vn, active)
    assert code == 0
    for l in range(cfg.n_layers):
        kp, vp = caches[l].k_pool.copy(), caches[l].v_pool.copy()
        new_len = oracle.kv_append(kp, vp, caches[l].page_table, lens, kn[l], vn[l], cfg.page_size,
                                   active=active.astype(bool))
        assert np.array_equal(support.to_host_bits(devs[l].k_pool, dtype), kp)
        assert np.array_equal(support.to_host_bits(devs[l].v_pool, dtype), vp)
    assert np.array_equal(devs[0].ctx_len.cpu().numpy(), new_len)


def test_capacity_overflow_is_reported_and_leaves_the_sequence_untouched():
    cfg = synth.CONFIGS["loop"].replace(B=2, n_layers=1)
    lens = np.array([120, 10], np.int32)
    caches = _layers(cfg, lens, 128, 1)                       # 2 pages: 128 slots per sequence
    kn, vn = synth.draw_new_block_kv(cfg, block=0, layer=0)
    devs, code = _append(cfg, caches, [kn], [vn])
    assert code == N.TT_ERR_CAPACITY
    assert list(devs[0].ctx_len.cpu().numpy()) == [120, 26]
    kp = caches[0].k_pool.copy()
    vp = caches[0].v_pool.copy()
    oracle.kv_append(kp, vp, caches[0].page_table, lens, kn, vn, cfg.page_size,
                     active=np.array([False, True]))
    assert np.array_equal(support.to_host_bits(devs[0].k_pool, "bf16"), kp)


def test_attention_after_append_matches_oracle():
    cfg = synth.CONFIGS["loop"].replace(B=3, n_layers=2, qkv_scale=1.0)
    lens = np.array([16384, 1000, 63], np.int32)
    caches = _layers(cfg, lens, 16384 + 64, cfg.n_layers, seed=2)
    kn, vn = zip(*[synth.draw_new_block_kv(cfg, block=0, layer=l) for l in range(cfg.n_layers)])
    devs, code = _append(cfg, caches, kn, vn)
    assert code == 0
    q, kb, vb = synth.draw_block_qkv(cfg, seed=2, block=1, layer=1)
    out = api.tt_denoise_attn(devs[1], *(support.to_dev(x, "bf16") for x in (q, kb, vb)))
    o = support.to_host_f64(out, "bf16")
    kp, vp = caches[1].k_pool.copy(), caches[1].v_pool.copy()
    new_len = oracle.kv_append(kp, vp, caches[1].page_table, lens, kn[1], vn[1], cfg.page_size)
    want, _ = oracle.denoise_attention(kp, vp, caches[1].page_table, new_len, cfg.page_size, q, kb, vb,
                                       1.0 / math.sqrt(cfg.D), "bf16")
    assert support.max_abs(o, want) <= 2e-2
