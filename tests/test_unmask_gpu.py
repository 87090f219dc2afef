"""Confidence unmasking on the GPU (tt_unmask) against the float64 oracle: commit masks
and token ids bit-exact outside the near-threshold band, confidences to 1e-5 relative."""
import numpy as np
import pytest
import torch

import oracle
from block_wise_diffusion_denoise_b300 import api, synth
from tests import support

pytestmark = pytest.mark.gpu


def _run_step(logits_bits, dtype, masked, tokens, tau, step, T, ws=None):
    B, S, V = logits_bits.shape
    lg = support.to_dev(logits_bits, dtype)
    m = torch.from_numpy(masked.astype(np.uint8)).cuda()
    t = torch.from_numpy(tokens.astype(np.int32)).cuda()
    com = torch.full((B, S), 7, dtype=torch.uint8, device="cuda")
    conf = torch.zeros((B, S), dtype=torch.float32, device="cuda")
    nm = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    err = api.error_word()
    api.tt_unmask(lg, m, t, tau, step, T, committed_now=com, conf=conf, n_masked=nm, ws=ws, dev_err=err)
    assert api.tt_get_device_error(err) == 0
    return (m.cpu().numpy(), t.cpu().numpy(), com.cpu().numpy(), conf.cpu().numpy(), nm.cpu().numpy())


def _check_step(logits_bits, dtype, masked, tokens, tau, step, T, ws=None, stats=None):
    g = _run_step(logits_bits, dtype, masked, tokens, tau, step, T, ws)
    ora = oracle.unmask(logits_bits, masked, tokens, tau, step, T, dtype)
    st = support.compare_unmask(masked, tokens, ora, *g, tau, step, T)
    if stats is not None:
        stats += st
    return g, ora, st


@pytest.fixture
def stats(request):
    """Counts of what the test's unmasking comparisons covered: reported at the end of the
    session and bounded here (at most 5 % of the sequences may differ from the float64
    decisions, and only inside the near-tau and fallback-tie bands)."""
    st = support.UnmaskStats()
    yield st
    support.report(request.node.name, st)
    st.check_bounds()


def test_tiny_fp32_block_loop(stats):
    cfg = synth.CONFIGS["tiny"]
    ws = api.workspace(api.tt_unmask_workspace_size(cfg.B, cfg.S, cfg.V, torch.float32))
    for blk in range(6):
        masked = np.ones((cfg.B, cfg.S), np.uint8)
        tokens = np.full((cfg.B, cfg.S), -1, np.int32)
        for step in range(1, cfg.T + 1):
            lg = synth.draw_logits(cfg, seed=blk, block=blk, step=step)
            (m, t, com, conf, nm), ora, _ = _check_step(lg, "f32", masked, tokens, cfg.tau, step, cfg.T, ws,
                                                        stats)
            assert com.sum() >= 1 or masked.sum() == 0
            masked, tokens = m, t
            if not masked.any():
                break
        assert not masked.any()        # every block finishes within T steps


@pytest.mark.parametrize("peak_hi", [12.0, 40.0])
def test_single_bf16_full_vocab(peak_hi, stats):
    cfg = synth.CONFIGS["single"]
    lg = synth.draw_logits(cfg, seed=3, peak_hi=peak_hi)
    masked = np.ones((cfg.B, cfg.S), np.uint8)
    tokens = np.full((cfg.B, cfg.S), -1, np.int32)
    for step in (1, cfg.T):
        _check_step(lg, "bf16", masked, tokens, cfg.tau, step, cfg.T, stats=stats)


@pytest.mark.parametrize("tau", [0.9, 0.8])
def test_batch_sharp_variant_every_branch(tau, stats):
    """B=32, V=131072; peaks U[0,40] in half the sequences and U[0,12] in the other half, so that
    the threshold, the fallback and step T all occur; at the workloads' threshold 0.9 and at the
    0.8 one of the pages' two-GPU runs."""
    cfg = synth.CONFIGS["ctx8k"].replace(tau=tau)
    rng = np.random.default_rng(11)
    ws = api.workspace(api.tt_unmask_workspace_size(cfg.B, cfg.S, cfg.V, torch.bfloat16))
    lg = synth.draw_logits(cfg, seed=5, peak_hi=40.0)
    lg[cfg.B // 2:] = synth.draw_logits(cfg, seed=6, peak_hi=12.0)[cfg.B // 2:]   # mild half: fallback
    masked = (rng.random((cfg.B, cfg.S)) < 0.8).astype(np.uint8)
    masked[:, 0] = 1
    tokens = np.where(masked == 1, -1, rng.integers(0, cfg.V, (cfg.B, cfg.S))).astype(np.int32)
    saw_thr = saw_fb = False
    for step in (1, 7, cfg.T):
        (m, t, com, conf, nm), ora, _ = _check_step(lg, "bf16", masked, tokens, cfg.tau, step, cfg.T, ws,
                                                    stats)
        if step < cfg.T:
            saw_fb |= any(r.fallback for r in ora)
            saw_thr |= any((r.committed_now.sum() > 0 and not r.fallback) for r in ora)
    assert saw_thr and saw_fb


def test_locked_rows_are_never_read_and_ties_take_lowest_id(stats):
    cfg = synth.CONFIGS["single"].replace(B=3, V=40000)
    lg = synth.draw_logits(cfg, seed=9, peak_hi=30.0)
    vals = oracle.decode(lg, "bf16")
    # exact ties at the maximum: copy the row maximum to a later and an earlier index
    for b in range(cfg.B):
        for p in range(0, cfg.S, 3):
            a = int(np.argmax(vals[b, p]))
            lg[b, p, min(cfg.V - 1, a + 17)] = lg[b, p, a]
            if a > 5:
                lg[b, p, a - 5] = lg[b, p, a]
    masked = np.ones((cfg.B, cfg.S), np.uint8)
    masked[:, 1::4] = 0
    tokens = np.where(masked == 1, -1, 123).astype(np.int32)
    lg_nan = lg.copy()
    lg_nan[masked == 0] = np.uint16(0x7FC0)          # NaN rows where positions are locked
    for step in (1, 2, cfg.T):
        g = _run_step(lg_nan, "bf16", masked, tokens, cfg.tau, step, cfg.T)
        ora = oracle.unmask(lg, masked, tokens, cfg.tau, step, cfg.T, "bf16")
        stats += support.compare_unmask(masked, tokens, ora, *g, cfg.tau, step, cfg.T)


@pytest.mark.parametrize("V", [1, 7, 8, 1003, 4100, 8200, 16384, 16385, 16392, 40000, 50001])
def test_ragged_vocab_sizes(V, stats):
    """Vocabulary sizes that are not a multiple of the vector width (unaligned rows: the chunked
    kernel) or of the streaming pass's 16 KB unit and 4-unit block (aligned rows: a partial last
    unit, a partial last block)."""
    for dtype in ("bf16", "f32"):
        cfg = synth.CONFIGS["tiny"].replace(B=2, V=V, dtype=dtype)
        lg = synth.draw_logits(cfg, seed=V, peak_hi=20.0)
        masked = np.ones((cfg.B, cfg.S), np.uint8)
        tokens = np.full((cfg.B, cfg.S), -1, np.int32)
        for step in (1, cfg.T):
            _check_step(lg, dtype, masked, tokens, cfg.tau, step, cfg.T, stats=stats)


def test_nothing_masked_and_empty_batch():
    cfg = synth.CONFIGS["tiny"].replace(B=2)
    lg = synth.draw_logits(cfg, seed=1)
    masked = np.zeros((cfg.B, cfg.S), np.uint8)
    tokens = np.arange(cfg.B * cfg.S, dtype=np.int32).reshape(cfg.B, cfg.S)
    m, t, com, conf, nm = _run_step(lg, "f32", masked, tokens, 0.9, 1, 4)
    assert not com.any() and np.array_equal(t, tokens) and (nm == 0).all() and np.isnan(conf).all()
    empty = torch.zeros((0, 16, 64), dtype=torch.float32, device="cuda")
    api.tt_unmask(empty, torch.zeros((0, 16), dtype=torch.uint8, device="cuda"),
                  torch.zeros((0, 16), dtype=torch.int32, device="cuda"), 0.9, 1, 4)
    torch.cuda.synchronize()


def test_batch_above_the_flag_snapshot(stats):
    """1100 sequences x 16 positions = 17600 rows, more than the 16384 masked flags the pass
    copies into shared memory: its producer and publisher read the flags from global memory."""
    cfg = synth.CONFIGS["single"].replace(B=1100, V=1024)
    rng = np.random.default_rng(11)
    lg = synth.draw_logits(cfg, seed=21, peak_hi=30.0)
    masked = (rng.random((cfg.B, cfg.S)) < 0.6).astype(np.uint8)
    masked[:5] = 0                                   # sequences with nothing masked
    masked[-3:] = 1
    tokens = np.where(masked == 1, -1, 5).astype(np.int32)
    for step in (1, cfg.T):
        _check_step(lg, "bf16", masked, tokens, cfg.tau, step, cfg.T, stats=stats)


def test_large_batch(stats):
    """260 sequences (4160 rows, more blocks than the grid has CTAs many times over); mixed
    masked rows, a few sequences with nothing masked, every branch of the rules."""
    cfg = synth.CONFIGS["single"].replace(B=260, V=4096)
    rng = np.random.default_rng(4)
    lg = synth.draw_logits(cfg, seed=13, peak_hi=30.0)
    masked = (rng.random((cfg.B, cfg.S)) < 0.7).astype(np.uint8)
    masked[:8] = 0                                   # a few sequences with nothing masked
    tokens = np.where(masked == 1, -1, 77).astype(np.int32)
    for step in (1, 5, cfg.T):
        _check_step(lg, "bf16", masked, tokens, cfg.tau, step, cfg.T, stats=stats)


@pytest.mark.parametrize("B", [31, 64])
def test_counters_are_left_zero_and_the_next_call_sees_every_block(B, stats):
    """The streaming pass hands the blocks of masked rows out from a counter in the workspace;
    the sequences' tickets and that counter must end every launch at zero (they are the
    workspace's last (B + 1) words, padded to 256 bytes), or the next call would skip blocks.
    Three calls on one workspace with different masks (a sequence with no masked row, rows
    masked at random, then every row), each checked against the oracle."""
    cfg = synth.CONFIGS["ctx8k"].replace(B=B, V=40000)   # two units per row, the second ragged
    ws = api.workspace(api.tt_unmask_workspace_size(cfg.B, cfg.S, cfg.V, torch.bfloat16))
    tail = ((B + 1) * 4 + 255) // 256 * 256
    rng = np.random.default_rng(B)
    for call in range(3):
        lg = synth.draw_logits(cfg, seed=40 + call, peak_hi=30.0)
        masked = (rng.random((cfg.B, cfg.S)) < 0.6).astype(np.uint8) if call < 2 else np.ones((cfg.B, cfg.S), np.uint8)
        if call == 0:
            masked[3] = 0
        tokens = np.where(masked == 1, -1, 5).astype(np.int32)
        _check_step(lg, "bf16", masked, tokens, cfg.tau, 2, cfg.T, ws, stats)
        torch.cuda.synchronize()
        assert int(ws[-tail:].abs().sum()) == 0, call


def test_no_masked_row_then_every_row_on_one_workspace(stats):
    """A call in which no row is masked hands out no block (the counter is never touched), and
    the next call on the same workspace, with every row masked, still reads every block."""
    cfg = synth.CONFIGS["ctx8k"].replace(B=8, V=70000)      # three units per row, two blocks
    ws = api.workspace(api.tt_unmask_workspace_size(cfg.B, cfg.S, cfg.V, torch.bfloat16))
    tail = ((cfg.B + 1) * 4 + 255) // 256 * 256
    lg = synth.draw_logits(cfg, seed=77, peak_hi=30.0)
    none = np.zeros((cfg.B, cfg.S), np.uint8)
    tokens = np.full((cfg.B, cfg.S), 9, np.int32)
    m, t, com, conf, nm = _run_step(lg, "bf16", none, tokens, cfg.tau, 3, cfg.T, ws)
    assert not m.any() and (t == 9).all() and not com.any() and np.isnan(conf).all() and (nm == 0).all()
    assert int(ws[-tail:].abs().sum()) == 0
    full = np.ones((cfg.B, cfg.S), np.uint8)
    _check_step(lg, "bf16", full, np.full((cfg.B, cfg.S), -1, np.int32), cfg.tau, 3, cfg.T, ws, stats)
    assert int(ws[-tail:].abs().sum()) == 0


def test_largest_batch_with_the_flag_copy(stats):
    """16384 rows (1024 x 16), the most the pass copies into shared memory: every CTA walks
    the flags far from its first rank and takes dozens of ranks from the counter.  Rows
    masked at random, small vocabulary; every sequence checked against the oracle."""
    cfg = synth.CONFIGS["ctx8k"].replace(B=1024, V=96)
    rng = np.random.default_rng(5)
    ws = api.workspace(api.tt_unmask_workspace_size(cfg.B, cfg.S, cfg.V, torch.bfloat16))
    lg = synth.draw_logits(cfg, seed=55, peak_hi=12.0)
    masked = (rng.random((cfg.B, cfg.S)) < 0.5).astype(np.uint8)
    masked[::7] = 0                                       # some sequences with nothing masked
    tokens = np.where(masked == 1, -1, 3).astype(np.int32)
    _check_step(lg, "bf16", masked, tokens, cfg.tau, 5, cfg.T, ws, stats)
    tail = ((cfg.B + 1) * 4 + 255) // 256 * 256
    assert int(ws[-tail:].abs().sum()) == 0
