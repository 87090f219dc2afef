"""Helpers of the GPU parity tests: move seeded inputs to the device and compare the
CUDA path's results with the float64 oracle."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
from block_wise_diffusion_denoise_b300 import synth
from block_wise_diffusion_denoise_b300.api import KVCache

TORCH_DT = {"bf16": torch.bfloat16, "f32": torch.float32}
NEAR_TAU = 1e-4          # oracle confidences this close to tau may commit on either side
CONF_REL = 1e-5          # the kernel's fp32 confidence against the float64 oracle (relative)
FALLBACK_TIE_REL = 2 * CONF_REL   # two confidences this close may be ordered either way in fp32


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


@dataclasses.dataclass
class UnmaskStats:
    """What one or more unmasking comparisons covered.

    sequences        sequences compared against the float64 oracle
    exact            of those, sequences whose decisions equal the oracle's bit for bit
    near_tau_seqs    sequences whose decisions differ only through positions whose oracle
                     confidence lies within NEAR_TAU of tau (either side is correct)
    fallback_tie_seqs  sequences where both sides took the at-least-one rule and picked
                     positions whose oracle confidences are within FALLBACK_TIE_REL
    positions        masked positions compared (confidence, argmax)
    near_tau_positions  masked positions inside the NEAR_TAU band
    rule_only        sequences without an oracle entry, checked by the rules alone
    """
    sequences: int = 0
    exact: int = 0
    near_tau_seqs: int = 0
    fallback_tie_seqs: int = 0
    positions: int = 0
    near_tau_positions: int = 0
    rule_only: int = 0

    def __iadd__(self, o):
        for f in dataclasses.fields(self):
            setattr(self, f.name, getattr(self, f.name) + getattr(o, f.name))
        return self

    def check_bounds(self, max_frac=0.05):
        """At most max_frac of the compared sequences (at least one) may differ from the oracle's
        float64 decisions, and then only inside the bands above."""
        differing = self.near_tau_seqs + self.fallback_tie_seqs
        assert self.sequences > 0 or self.rule_only > 0, "nothing was compared"
        assert differing <= max(1, int(max_frac * self.sequences)), self
        assert self.near_tau_positions <= max(1, int(max_frac * self.positions)), self


REPORT = {}   # test id -> UnmaskStats, printed at the end of the session (tests/conftest.py)


def report(name: str, stats: UnmaskStats) -> UnmaskStats:
    REPORT.setdefault(name, UnmaskStats())
    REPORT[name] += stats
    return stats


def compare_unmask(pre_masked, pre_tokens, ora, gpu_masked, gpu_tokens, gpu_committed, gpu_conf,
                   gpu_nmasked, tau, step, T) -> UnmaskStats:
    """Comparison of one unmasking step, sequence by sequence.

    Every sequence, with or without an oracle entry: only masked positions commit, locked
    ones never change, the mask and the count left follow the commits, confidences are NaN
    exactly at locked positions, and the committed set is exactly the commit rule applied to
    the kernel's own fp32 confidences (the decision taken in the kernel's precision).

    With an oracle entry (float64): the token of every committed position is the oracle's
    argmax (exact on both sides), every masked confidence is within CONF_REL of the oracle's,
    and the committed set equals the oracle's, except where floating point legitimately
    decides it differently -- a position whose oracle confidence is within NEAR_TAU of tau, or
    a fallback choice between positions whose oracle confidences are within FALLBACK_TIE_REL.
    Those cases are counted, never silently dropped.  Returns the counts."""
    B, S = pre_masked.shape
    st = UnmaskStats()
    for b in range(B):
        r = ora[b]
        m0 = pre_masked[b].astype(bool)
        com = gpu_committed[b].astype(bool)
        conf = gpu_conf[b].astype(np.float64)
        # ---- checks that need no float64 oracle
        assert not (com & ~m0).any(), (b, "committed a locked position")
        assert np.array_equal(gpu_tokens[b][~m0], pre_tokens[b][~m0]), (b, "a locked token changed")
        assert np.array_equal(gpu_masked[b].astype(bool), m0 & ~com), b
        assert gpu_nmasked[b] == int((m0 & ~com).sum()), b
        assert np.isnan(conf[~m0]).all() and np.isfinite(conf[m0]).all(), b
        assert (conf[m0] > 0).all() and (conf[m0] <= 1.0 + 1e-6).all(), b
        want_com, _ = oracle.commit_rule(conf, m0, tau, step, T)
        assert np.array_equal(com, want_com), (b, "the rule on the kernel's confidences", com, want_com)
        assert (gpu_tokens[b][com] >= 0).all(), b
        if r is None:
            st.rule_only += 1
            continue
        # ---- against the float64 oracle
        st.sequences += 1
        for p in np.nonzero(com)[0]:
            assert gpu_tokens[b, p] == r.argmax[p], (b, p, gpu_tokens[b, p], r.argmax[p])
        if m0.any():
            rel = np.abs(conf[m0] - r.conf[m0]) / r.conf[m0]
            assert rel.max() < CONF_REL, (b, rel.max())
        rconf = np.nan_to_num(r.conf, nan=-1.0)
        near = m0 & (np.abs(rconf - tau) < NEAR_TAU)
        st.positions += int(m0.sum())
        st.near_tau_positions += int(near.sum())
        if np.array_equal(com, r.committed_now):
            st.exact += 1
            continue
        diff = com != r.committed_now
        gpu_fb = oracle.commit_rule(conf, m0, tau, step, T)[1]
        clear_above = m0 & ~near & (rconf >= tau)
        if not (diff & ~near).any():
            st.near_tau_seqs += 1              # only near-tau positions went the other way
        elif near.any() and not clear_above.any() and (gpu_fb or r.fallback):
            st.near_tau_seqs += 1              # near-tau positions decided whether the fallback ran
        elif gpu_fb and r.fallback and diff.sum() == 2:
            pg, po = int(np.nonzero(com)[0][0]), int(np.nonzero(r.committed_now)[0][0])
            assert rconf[pg] >= rconf[po] * (1.0 - FALLBACK_TIE_REL), (b, pg, po, rconf[pg], rconf[po])
            st.fallback_tie_seqs += 1
        else:
            raise AssertionError((b, "commit sets differ outside the near-tau and fallback-tie bands",
                                  com, r.committed_now, r.conf))
    return st
