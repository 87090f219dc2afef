"""The scratch-free unmasking entry point (tt_unmask_noalloc).

It serves callers that cannot allocate device memory -- code running under CUDA
graph capture, plugins inside a framework that owns the whole device pool, and
real-time loops with memory fixed at start-up -- by keeping its scratch in the
library's own file-scope device array.  These tests call it through the C ABI and
require exactly the results of tt_unmask (which takes a caller workspace) on two
calls in a row, the second one reusing whatever the first left in the array.

This file is named to be collected last, so a run that stops at the first failure
has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from block_wise_diffusion_denoise_b300 import _native as N
from block_wise_diffusion_denoise_b300 import api, synth
from tests import support


def _state(cfg, seed):
    rng = np.random.default_rng(seed)
    masked = (rng.random((cfg.B, cfg.S)) < 0.75).astype(np.uint8)
    masked[:, 0] = 1
    tokens = np.where(masked == 1, -1, rng.integers(0, cfg.V, (cfg.B, cfg.S))).astype(np.int32)
    return masked, tokens


def _outputs(cfg, dtype, lg_dev, masked, tokens, step, noalloc):
    m = torch.from_numpy(masked).cuda()
    t = torch.from_numpy(tokens).cuda()
    com = torch.full((cfg.B, cfg.S), 9, dtype=torch.uint8, device="cuda")
    conf = torch.zeros((cfg.B, cfg.S), dtype=torch.float32, device="cuda")
    nm = torch.full((cfg.B,), -1, dtype=torch.int32, device="cuda")
    err = api.error_word()
    if noalloc:
        api.tt_unmask_noalloc(lg_dev, m, t, cfg.tau, step, cfg.T, committed_now=com, conf=conf, n_masked=nm,
                              dev_err=err)
    else:
        api.tt_unmask(lg_dev, m, t, cfg.tau, step, cfg.T, committed_now=com, conf=conf, n_masked=nm, dev_err=err)
    assert api.tt_get_device_error(err) == 0
    return [x.cpu().numpy() for x in (m, t, com, conf, nm)]


@pytest.mark.gpu
@pytest.mark.parametrize("name,dtype", [("ctx8k", "bf16"), ("tiny", "f32"), ("large_batch", "f32")])
def test_noalloc_matches_workspace_entry_point_twice(name, dtype):
    """ctx8k: full vocabulary; tiny: fp32; large_batch: 260 sequences x 16 positions at V = 1024,
    many more blocks than CTAs."""
    if name == "large_batch":
        cfg = synth.CONFIGS["single"].replace(B=260, V=1024, dtype=dtype)
    else:
        cfg = synth.CONFIGS[name].replace(dtype=dtype)
    lg = synth.draw_logits(cfg, seed=21, peak_hi=40.0)
    if cfg.B > 1:
        lg[cfg.B // 2:] = synth.draw_logits(cfg, seed=22, peak_hi=12.0)[cfg.B // 2:]
    lg_dev = support.to_dev(lg, dtype)
    masked, tokens = _state(cfg, 3)
    for step in (1, 2):                       # two calls in a row; the second reuses the array
        want = _outputs(cfg, dtype, lg_dev, masked, tokens, step, noalloc=False)
        got = _outputs(cfg, dtype, lg_dev, masked, tokens, step, noalloc=True)
        for w, g in zip(want, got):
            assert np.array_equal(w, g, equal_nan=True)
        masked, tokens = got[0], got[1]


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """A shape whose scratch would not fit the array is refused on the host, before any launch."""
    lib = N.lib()
    need = ctypes.c_size_t(0)
    assert lib.tt_unmask_workspace_size(64, 64, 131072, N.TT_BF16, ctypes.byref(need)) == N.TT_OK
    assert need.value > N.UNMASK_NOALLOC_SCRATCH_BYTES
    st = lib.tt_unmask_noalloc(0x10000, N.TT_BF16, 64, 64, 131072, 0.9, 1, 4, 0x20000, 0x30000, None, None,
                               None, None, None)
    assert st == N.TT_ERR_CAPACITY
