"""The masked-diffusion objective on the GPU against the float64 oracle: the linear-schedule
corruption (tt_linear_schedule_mask) bit for bit, and the masked NLL (tt_masked_nll) per
position within 1e-5 * max(1, |nll|), with the per-sequence sums and counts.

Definitions: TwoTower summary on gist.science, "Training und Konditionierung -- Maskierte
Diffusion" (corruption of clean blocks under a linear schedule; NLL of the original tokens
at the masked positions)."""
import numpy as np
import pytest
import torch

import oracle
from block_wise_diffusion_denoise_b300 import _native as N
from block_wise_diffusion_denoise_b300 import api, synth
from tests import support

pytestmark = pytest.mark.gpu

NLL_TOL = 1e-5     # |nll_gpu - nll_oracle| <= NLL_TOL * max(1, |nll_oracle|)


def _corrupt(clean, u, t, mask_id=-7):
    d = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x)).to(dt).cuda()   # noqa: E731
    masked = torch.full(u.shape, 9, dtype=torch.uint8, device="cuda")
    noisy = torch.full(u.shape, 12345, dtype=torch.int32, device="cuda")
    err = api.error_word()
    api.tt_linear_schedule_mask(d(u, torch.float32), d(t, torch.float32), masked=masked,
                                clean=d(clean, torch.int32), mask_id=mask_id, noisy=noisy, dev_err=err)
    code = api.tt_get_device_error(err)
    return masked.cpu().numpy(), noisy.cpu().numpy(), code


def test_linear_schedule_bit_exact():
    cfg = synth.CONFIGS["ctx8k"]
    clean, u, t = synth.draw_corruption(cfg, seed=1)
    t[:4] = [0.0, 1.0, np.float32(0.5), u[3, 5]]       # endpoints and a tie u == t (not masked)
    masked, noisy, code = _corrupt(clean, u, t)
    assert code == 0
    for b in range(cfg.B):
        want = oracle.linear_schedule_mask(u[b], float(t[b]))
        assert np.array_equal(masked[b].astype(bool), want), b
        assert np.array_equal(noisy[b], np.where(want, -7, clean[b])), b
    assert not masked[0].any() and masked[1].all() and not masked[3, 5]


def test_linear_schedule_rejects_times_outside_the_unit_interval():
    cfg = synth.CONFIGS["tiny"].replace(B=3)
    clean, u, t = synth.draw_corruption(cfg, seed=2)
    t[1] = 1.5
    masked, noisy, code = _corrupt(clean, u, t)
    assert code == N.TT_ERR_BOUNDS
    assert (masked[1] == 9).all() and (noisy[1] == 12345).all()          # untouched
    for b in (0, 2):
        assert np.array_equal(masked[b].astype(bool), oracle.linear_schedule_mask(u[b], float(t[b])))


def _nll_case(lg_bits, dtype, targets, masked):
    B, S, V = lg_bits.shape
    lg = support.to_dev(lg_bits, dtype)
    err = api.error_word()
    ws = api.workspace(api.tt_masked_nll_workspace_size(B, S, V, support.TORCH_DT[dtype]))
    outs = []
    for _ in range(2):                                 # twice: the workspace is left reusable
        nll, tot, cnt = api.tt_masked_nll(lg, torch.from_numpy(targets.astype(np.int32)).cuda(),
                                          torch.from_numpy(masked.astype(np.uint8)).cuda(), ws=ws, dev_err=err)
        assert api.tt_get_device_error(err) == 0
        outs.append((nll.cpu().numpy(), tot.cpu().numpy(), cnt.cpu().numpy()))
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b, equal_nan=True)     # deterministic
    return outs[0]


def _check_nll(lg_bits, dtype, targets, masked):
    nll, tot, cnt = _nll_case(lg_bits, dtype, targets, masked)
    w_nll, w_tot, w_cnt = oracle.masked_nll(lg_bits, targets, masked, dtype)
    m = masked.astype(bool)
    assert np.isnan(nll[~m]).all()
    err = np.abs(nll[m] - w_nll[m]) / np.maximum(1.0, np.abs(w_nll[m]))
    assert err.max(initial=0.0) <= NLL_TOL, err.max()
    assert np.array_equal(cnt, w_cnt)
    # the sum of S values, each within the bound above, plus fp32 rounding of the sum
    bound = NLL_TOL * np.maximum(1.0, np.abs(np.where(m, w_nll, 0)).sum(axis=1)) + 1e-6 * np.abs(w_tot)
    assert (np.abs(tot - w_tot) <= bound + 1e-6).all(), np.abs(tot - w_tot).max()
    return nll, w_nll


@pytest.mark.parametrize("peak_hi", [12.0, 40.0])
def test_masked_nll_full_vocab(peak_hi):
    """The ctx8k batch shape (32 x 16 positions, V = 131072, bf16), masks from the linear
    schedule at per-sequence times, half the targets at the row's argmax (small NLL)."""
    cfg = synth.CONFIGS["ctx8k"]
    lg = synth.draw_logits(cfg, seed=31, peak_hi=peak_hi)
    clean, u, t = synth.draw_corruption(cfg, seed=31)
    t[0], t[1] = 0.0, 1.0                               # a sequence with nothing masked, one all masked
    masked = np.stack([oracle.linear_schedule_mask(u[b], float(t[b])) for b in range(cfg.B)])
    vals = oracle.decode(lg, "bf16")
    targets = np.where(np.arange(cfg.S)[None, :] % 2 == 0, vals.argmax(axis=2), clean).astype(np.int32)
    _check_nll(lg, "bf16", targets, masked)


@pytest.mark.parametrize("V,dtype", [(1024, "f32"), (8, "bf16"), (8200, "bf16"), (40000, "bf16"),
                                     (4100, "f32"), (16392, "f32")])
def test_masked_nll_vocab_sizes(V, dtype):
    cfg = synth.CONFIGS["tiny"].replace(B=5, V=V, dtype=dtype)
    lg = synth.draw_logits(cfg, seed=V, peak_hi=20.0)
    clean, u, t = synth.draw_corruption(cfg, seed=V)
    masked = np.stack([oracle.linear_schedule_mask(u[b], float(t[b])) for b in range(cfg.B)])
    masked[0] = True
    _check_nll(lg, dtype, clean, masked)


def test_masked_nll_special_rows():
    """All logits equal (NLL = log V exactly in the definition), very large and very negative
    logits (|l| up to 1e37), a dominant target (NLL far below 1e-5), and exact ties."""
    B, S, V = 2, 16, 131072
    rng = np.random.default_rng(5)
    x = rng.normal(0, 3, size=(B, S, V)).astype(np.float32)
    x[0, 0] = 7.25                                     # all equal
    x[0, 1] = 1e37 + rng.normal(0, 1e35, size=V).astype(np.float32)     # huge, spread
    x[0, 2] = -1e37 + rng.normal(0, 1e35, size=V).astype(np.float32)
    x[0, 3, 100] = 60.0                                # dominant target (NLL ~ V e^-60)
    x[0, 4, [5, 77, 9000]] = 30.0                      # three-way tie at the maximum
    targets = rng.integers(0, V, size=(B, S)).astype(np.int32)
    targets[0, 3] = 100
    targets[0, 4] = 77
    masked = np.ones((B, S), bool)
    masked[1, ::3] = False
    for dtype in ("f32", "bf16"):
        lg = synth.bf16_bits(x) if dtype == "bf16" else x
        nll, want = _check_nll(lg, dtype, targets, masked)
        assert abs(nll[0, 0] - np.log(V)) <= NLL_TOL * np.log(V)
        assert 0.0 <= nll[0, 3] < 1e-6


def test_masked_nll_large_batch_and_bad_target():
    cfg = synth.CONFIGS["single"].replace(B=300, V=2048)
    lg = synth.draw_logits(cfg, seed=8, peak_hi=15.0)
    clean, u, t = synth.draw_corruption(cfg, seed=8)
    masked = np.stack([oracle.linear_schedule_mask(u[b], float(t[b])) for b in range(cfg.B)])
    _check_nll(lg, "bf16", clean, masked)
    # a masked position whose target lies outside the vocabulary: NaN there, the error word set
    bad = clean.copy()
    masked[3, 2] = True
    bad[3, 2] = cfg.V
    err = api.error_word()
    nll, tot, cnt = api.tt_masked_nll(support.to_dev(lg, "bf16"), torch.from_numpy(bad).cuda(),
                                      torch.from_numpy(masked.astype(np.uint8)).cuda(), dev_err=err)
    assert api.tt_get_device_error(err) == N.TT_ERR_BOUNDS
    nll = nll.cpu().numpy()
    assert np.isnan(nll[3, 2]) and np.isnan(tot.cpu().numpy()[3])
    assert np.isfinite(nll[4][masked[4]]).all()


def test_masked_nll_batch_above_the_flag_snapshot():
    """17600 rows, more than the 16384 masked flags the pass copies into shared memory."""
    cfg = synth.CONFIGS["single"].replace(B=1100, V=1024)
    lg = synth.draw_logits(cfg, seed=9, peak_hi=15.0)
    clean, u, t = synth.draw_corruption(cfg, seed=9)
    masked = np.stack([oracle.linear_schedule_mask(u[b], float(t[b])) for b in range(cfg.B)])
    _check_nll(lg, "bf16", clean, masked)


def test_masked_nll_rejects_unaligned_rows():
    lg = torch.zeros((2, 16, 1003), dtype=torch.bfloat16, device="cuda")
    m = torch.ones((2, 16), dtype=torch.uint8, device="cuda")
    tg = torch.zeros((2, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(api.TTError) as e:
        api.tt_masked_nll(lg, tg, m)
    assert e.value.status == N.TT_ERR_UNSUPPORTED


def test_counters_are_left_zero_between_calls():
    """The tickets and the block counter of the streaming pass (the workspace's last (B + 1)
    words, padded to 256 bytes) are zero after every call; a second call on the same
    workspace with another mask still reads every masked row."""
    B, S, V = 40, 16, 40000
    cfg = synth.CONFIGS["ctx8k"].replace(B=B, V=V)
    lg = synth.draw_logits(cfg, seed=8, peak_hi=25.0)
    rng = np.random.default_rng(8)
    targets = rng.integers(0, V, (B, S)).astype(np.int32)
    dev = support.to_dev(lg, "bf16")
    err = api.error_word()
    ws = api.workspace(api.tt_masked_nll_workspace_size(B, S, V, torch.bfloat16))
    tail = ((B + 1) * 4 + 255) // 256 * 256
    for call in range(2):
        masked = (rng.random((B, S)) < (0.3 if call == 0 else 0.9)).astype(np.uint8)
        nll, tot, cnt = api.tt_masked_nll(dev, torch.from_numpy(targets).cuda(), torch.from_numpy(masked).cuda(),
                                          ws=ws, dev_err=err)
        assert api.tt_get_device_error(err) == 0
        w_nll, w_tot, w_cnt = oracle.masked_nll(lg, targets, masked, "bf16")
        got = nll.cpu().numpy()
        sel = masked == 1
        assert np.array_equal(cnt.cpu().numpy(), w_cnt)
        assert np.all(np.abs(got[sel] - w_nll[sel]) <= NLL_TOL * np.maximum(1.0, np.abs(w_nll[sel])))
        assert np.isnan(got[~sel]).all()
        torch.cuda.synchronize()
        assert int(ws[-tail:].abs().sum()) == 0, call
