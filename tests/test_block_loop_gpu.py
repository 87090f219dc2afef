"""The full block loop through the C ABI, in lockstep with the float64 oracle: every step
runs tt_block_step (the attention of every layer, then the unmasking of the step's logits),
every finished block is committed with tt_kv_append, and the next block attends to the
grown caches.  Each oracle step starts from the GPU's state before the step, so a decision
inside the near-threshold band cannot cascade."""
import math

import numpy as np
import pytest
import torch

import oracle
from block_wise_diffusion_denoise_b300 import api, synth
from tests import support

pytestmark = pytest.mark.gpu


def _run_loop(cfg, lens, seed, peak_hi, sample=None, name="block loop"):
    """Runs the loop; checks everything against the oracle, or with ``sample`` (a function of
    (block, step) returning ([(layer, sequence), ...] for attention, [sequence, ...] for the
    unmasking)) only those, plus the rules' oracle-free checks on every sequence."""
    L = cfg.n_layers
    cap = int(lens.max()) + cfg.S * (cfg.n_blocks + 1)
    caches = [synth.draw_paged_cache(cfg, lens, cap, seed=seed, layer=l) for l in range(L)]
    devs = [support.cache_to_dev(c) for c in caches]
    for d in devs[1:]:
        d.ctx_len = devs[0].ctx_len                      # the layers hold the same tokens
    kp = [c.k_pool for c in caches]                      # the oracle's copy of every layer's cache
    vp = [c.v_pool for c in caches]                      # (the device holds its own copy)
    ctx = caches[0].ctx_len.copy()
    scale = 1.0 / math.sqrt(cfg.D)
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    ws = api.workspace(api.tt_block_step_workspace_size(cfg.B, cfg.S, cfg.Hq, cfg.Hkv, cfg.D, cfg.V, tdt))
    err = api.error_word()
    steps_run = 0
    stats = support.UnmaskStats()
    for blk in range(cfg.n_blocks):
        masked = torch.ones((cfg.B, cfg.S), dtype=torch.uint8, device="cuda")
        tokens = torch.full((cfg.B, cfg.S), -1, dtype=torch.int32, device="cuda")
        for step in range(1, cfg.T + 1):
            qkv = [synth.draw_block_qkv(cfg, seed=seed, block=blk, step=step, layer=l) for l in range(L)]
            lg = synth.draw_logits(cfg, seed=seed, block=blk, step=step, peak_hi=peak_hi)
            outs = [torch.empty((cfg.B, cfg.S, cfg.Hq, cfg.D), dtype=tdt, device="cuda") for _ in range(L)]
            com = torch.zeros((cfg.B, cfg.S), dtype=torch.uint8, device="cuda")
            conf = torch.zeros((cfg.B, cfg.S), dtype=torch.float32, device="cuda")
            nm = torch.zeros((cfg.B,), dtype=torch.int32, device="cuda")
            pre_m, pre_t = masked.cpu().numpy().copy(), tokens.cpu().numpy().copy()
            api.tt_block_step(devs, [support.to_dev(x[0], cfg.dtype) for x in qkv],
                              [support.to_dev(x[1], cfg.dtype) for x in qkv],
                              [support.to_dev(x[2], cfg.dtype) for x in qkv], outs,
                              support.to_dev(lg, cfg.dtype), masked, tokens, cfg.tau, step, cfg.T,
                              sm_scale=scale, committed_now=com, conf=conf, n_masked=nm, ws=ws, dev_err=err)
            assert api.tt_get_device_error(err) == 0
            # attention against the oracle on the current caches (every layer and sequence, or
            # the sampled ones)
            tol = 2e-2 if cfg.dtype == "bf16" else 1e-5
            if sample is None:
                attn_pairs, unmask_seqs = [(l, None) for l in range(L)], None
            else:
                attn_pairs, unmask_seqs = sample(blk, step)
            for l, b in attn_pairs:
                want, _ = oracle.denoise_attention(kp[l], vp[l], caches[l].page_table, ctx, cfg.page_size,
                                                   qkv[l][0], qkv[l][1], qkv[l][2], scale, cfg.dtype,
                                                   seqs=None if b is None else [b])
                got = support.to_host_f64(outs[l], cfg.dtype)
                if b is None:
                    assert support.max_abs(got, want) <= tol, (blk, step, l)
                else:
                    assert support.max_abs(got[b], want[b]) <= tol, (blk, step, l, b)
            # the unmasking against the oracle from the GPU's pre-step state
            ora = oracle.unmask(lg, pre_m, pre_t, cfg.tau, step, cfg.T, cfg.dtype, seqs=unmask_seqs)
            stats += support.compare_unmask(pre_m, pre_t, ora, masked.cpu().numpy(), tokens.cpu().numpy(),
                                            com.cpu().numpy(), conf.cpu().numpy(), nm.cpu().numpy(), cfg.tau,
                                            step, cfg.T)
            steps_run += 1
            if not masked.any():
                break
        assert not masked.any()                          # every block finishes within T steps
        # commit: the block's K/V of every layer joins that layer's context
        kv = [synth.draw_new_block_kv(cfg, seed=seed, block=blk, layer=l) for l in range(L)]
        api.tt_kv_append(devs, [support.to_dev(k, cfg.dtype) for k, _ in kv],
                         [support.to_dev(v, cfg.dtype) for _, v in kv], dev_err=err)
        assert api.tt_get_device_error(err) == 0
        for l in range(L):
            new_ctx = oracle.kv_append(kp[l], vp[l], caches[l].page_table, ctx, kv[l][0], kv[l][1],
                                       cfg.page_size)
        ctx = new_ctx
        assert np.array_equal(devs[0].ctx_len.cpu().numpy(), ctx)
    support.report(name, stats)
    stats.check_bounds()
    return steps_run


@pytest.mark.parametrize("peak_hi", [12.0, 40.0])
def test_block_loop_bf16_in_lockstep(peak_hi):
    """The loop workload's structure at a size the oracle runs in seconds: 3 sequences of
    ragged context, 3 attention layers, T=4, 3 blocks, V=8192."""
    cfg = synth.CONFIGS["loop"].replace(B=3, n_layers=3, T=4, n_blocks=3, V=8192, len_lo=100, len_hi=700)
    lens = np.array([100, 420, 700], np.int32)
    assert _run_loop(cfg, lens, seed=3, peak_hi=peak_hi, name=f"block loop bf16 peak {peak_hi}") >= cfg.n_blocks


def test_full_size_block_loop_sampled():
    """The loop workload at its full size -- 16 sequences of 16384 context tokens, 6 attention
    layers with their own caches, T = 16, 8 consecutive blocks, V = 131072 -- through the C ABI.
    At every step one (layer, sequence) attention segment and the unmasking of two sequences
    are checked against the oracle; every sequence gets the rules' oracle-free checks, every
    block must finish within T steps, and the lengths grow by one block per commit."""
    cfg = synth.CONFIGS["loop"]
    lens = synth.draw_lengths(cfg, 0)

    def sample(blk, step):
        i = blk * cfg.T + step
        return [(i % cfg.n_layers, (7 * i) % cfg.B)], sorted({(5 * i) % cfg.B, (5 * i + 3) % cfg.B})

    assert _run_loop(cfg, lens, seed=11, peak_hi=12.0, sample=sample, name="block loop full size") >= cfg.n_blocks


def test_block_loop_fp32_in_lockstep():
    cfg = synth.CONFIGS["tiny"].replace(B=2, n_layers=2, n_blocks=2, T=4)
    lens = np.array([64, 5], np.int32)
    assert _run_loop(cfg, lens, seed=4, peak_hi=None, name="block loop fp32") >= cfg.n_blocks
