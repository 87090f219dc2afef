"""Failure paths on the GPU, without faulting or hanging it: a bounded wait that can never
finish reports TT_ERR_DEVICE_TIMEOUT and leaves the context usable; kernels write nothing
outside their output buffers."""
import math

import numpy as np
import pytest
import torch

from block_wise_diffusion_denoise_b300 import api, synth
from block_wise_diffusion_denoise_b300 import _native as N
from tests import support

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports():
    err = api.error_word()
    api.tt_check_wait_timeout(2000, err)
    assert api.tt_get_device_error(err) == N.TT_ERR_DEVICE_TIMEOUT
    # the context is still usable: a normal call afterwards succeeds with a clean word
    cfg = synth.CONFIGS["tiny"]
    lg = support.to_dev(synth.draw_logits(cfg, seed=1), "f32")
    masked = torch.ones((cfg.B, cfg.S), dtype=torch.uint8, device="cuda")
    tokens = torch.full((cfg.B, cfg.S), -1, dtype=torch.int32, device="cuda")
    err2 = api.error_word()
    api.tt_unmask(lg, masked, tokens, cfg.tau, 1, cfg.T, dev_err=err2)
    assert api.tt_get_device_error(err2) == 0
    assert int(masked.sum()) < cfg.S


def test_attention_writes_only_its_output_rows():
    """The output lives inside a larger buffer whose guard rows hold a canary pattern."""
    cfg = synth.CONFIGS["ragged"].replace(B=4)
    cache, q, kb, vb = support.attention_case(cfg, seed=5)
    dev = support.cache_to_dev(cache)
    qd, kd, vd = (support.to_dev(x, "bf16") for x in (q, kb, vb))
    guard = 64
    big = torch.full((cfg.B * cfg.S * cfg.Hq * cfg.D + 2 * guard,), -12345, dtype=torch.int16, device="cuda")
    out = big[guard:guard + cfg.B * cfg.S * cfg.Hq * cfg.D].view(torch.bfloat16).view(cfg.B, cfg.S, cfg.Hq, cfg.D)
    api.tt_denoise_attn(dev, qd, kd, vd, out=out, sm_scale=1.0 / math.sqrt(cfg.D))
    torch.cuda.synchronize()
    b = big.cpu().numpy()
    assert (b[:guard] == -12345).all() and (b[-guard:] == -12345).all()
    assert not (b[guard:-guard] == -12345).all()


def test_unmask_writes_only_its_rows():
    cfg = synth.CONFIGS["single"].replace(B=3, V=20000)
    lg = support.to_dev(synth.draw_logits(cfg, seed=8, peak_hi=30.0), "bf16")
    n = cfg.B * cfg.S
    tok_big = torch.full((n + 64,), 777, dtype=torch.int32, device="cuda")
    msk_big = torch.full((n + 64,), 9, dtype=torch.uint8, device="cuda")
    tokens = tok_big[32:32 + n].view(cfg.B, cfg.S)
    masked = msk_big[32:32 + n].view(cfg.B, cfg.S)
    tokens.fill_(-1)
    masked.fill_(1)
    api.tt_unmask(lg, masked, tokens, cfg.tau, 1, cfg.T)
    torch.cuda.synchronize()
    t, m = tok_big.cpu().numpy(), msk_big.cpu().numpy()
    assert (t[:32] == 777).all() and (t[-32:] == 777).all()
    assert (m[:32] == 9).all() and (m[-32:] == 9).all()
    assert (m[32:-32] <= 1).all() and m[32:-32].sum() < n
