"""Float64 CPU oracle for one TwoTower denoiser step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import or call this
module; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA library: it decodes its
own inputs, reads the paged cache through the page table itself and applies
the definitions below with plain NumPy float64 arithmetic (a matrix product,
``exp`` and ``argmax`` are the only library primitives used).

Sources (the pages print no algorithm listing for these steps, only prose):

* [A] "Nemotron-TwoTower: Diffusion Language Modeling with Pretrained
  Autoregressive Context", AI summary on gist.science (German), section
  "Technisches Resümee — Architektur": the denoiser uses bidirectional block
  attention inside the noisy block and causal, layer-aligned cross-attention
  to the frozen context tower's KV for the same layer.
* [G] same page, "Technisches Resümee — Generierungsprozess" (Algorithm 1):
  a block starts as S masked tokens, is refined over T steps, and at every
  step the denoiser attends to the context tower's KV cache of past blocks and
  to its own bidirectional KV of the current block; a finished block is
  committed and the context tower extends its state with the clean tokens.
* [U] same page, "Training und Konditionierung — Sampling" (Algorithm 2):
  at each step all masked tokens are predicted in parallel, tokens whose
  confidence is above a threshold gamma are committed, the others stay masked.
  Also "Der Konfidenz-Trick": a confident word is locked at once and never
  revisited; an uncertain one stays masked for the next round.
* [T] same page, "Training und Konditionierung — Maskierte Diffusion": clean
  blocks are corrupted by replacing tokens with [MASK] following a linear
  schedule, and the denoiser minimises the negative log-likelihood of the
  original tokens at the masked positions.
* [R] dgnews.ru news article on Nemotron-TwoTower, section "How the
  architecture actually works": inside a block every masked position attends
  to all other block positions; towards earlier blocks and the prompt the
  attention stays causal; each denoiser layer reads the matching layer of the
  frozen context tower.

Readings where the pages are silent (each is listed with its reason in the
repository's design notes): the softmax scale is an argument (default
1/sqrt(D)); GQA head h reads KV head floor(h / G); every context position
precedes the block, so "causal" towards the context admits all L keys; no
mask inside the block for the denoiser, while the context tower, taking in a
committed block, lets block position i see block positions 0..i (its causal
order applied within the block); no positional logic (q and k arrive position-encoded);
confidence is the maximum softmax probability at temperature 1; a position is
committed when conf >= tau; if none qualifies the single most confident
masked position is committed (lowest position on ties); at step T every
masked position is committed; argmax ties resolve to the lowest token id.
On the training side, the linear schedule masks each position independently
with probability t (it survives with probability 1 - t), the uniform draws are
inputs, and the loss is the per-position NLL of the clean token at the masked
positions with its sum and count per sequence (no weight over t: the pages
state none).

Parity of every function here is pinned by ``tests/test_oracle_pins.py``
(brute force, closed forms, a library routine for the no-context case, and
invariants); no function is "parity unpinned".
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np


# --------------------------------------------------------------------------- decoding

def decode(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of each stored element (bf16 bit patterns or float32)."""
    if dtype == "bf16":
        bits = np.asarray(x).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype}")


# --------------------------------------------------------------------------- context KV

def context_rows(pool: np.ndarray, page_table_row: np.ndarray, L: int, page_size: int) -> np.ndarray:
    """The first L context positions of one sequence, in logical order.

    Position j lives in page ``page_table_row[j // page_size]`` at slot
    ``j % page_size``.  ``pool`` is [num_pages, Hkv, page_size, D]; the result is
    [L, Hkv, D].  Slots at or beyond L are never touched.
    """
    j = np.arange(L)
    pages = np.asarray(page_table_row)[j // page_size]
    slots = j % page_size
    return pool[pages, :, slots, :]


# --------------------------------------------------------------------------- attention

def denoise_attention_seq(q: np.ndarray, k_ctx: np.ndarray, v_ctx: np.ndarray,
                          k_blk: np.ndarray, v_blk: np.ndarray, sm_scale: float,
                          key_bias: Optional[np.ndarray] = None, return_probs: bool = False,
                          causal_block: bool = False):
    """Two-segment attention of one sequence's block queries ([A], [G], [R]).

    q [S, Hq, D]; k_ctx, v_ctx [L, Hkv, D] (context tower KV of this layer, L may
    be 0); k_blk, v_blk [S, Hkv, D] (the block's own KV).  Query head h reads
    KV head g = h // (Hq // Hkv).  Each block query sees every context key and
    every block key (bidirectional inside the block, no mask):

        s_j = sm_scale * <q_{i,h}, k_{j,g}>     for j over [context ; block]
        p   = softmax(s)                        (over all L + S keys)
        o_{i,h} = sum_j p_j v_{j,g}

    With ``causal_block`` the block is read the way the frozen context tower
    reads it when it takes in a committed block ([A]: that tower is a causal
    autoregressive model over the prompt and the committed tokens; [G]: after a
    commit it extends its state with the clean block): block query i still sees
    every context key, but of the block keys only j <= i.

    ``key_bias`` (optional, [L + S]) is added to every score of the key; -inf
    removes a key.  Returns o [S, Hq, D] and lse [Hq, S] = log sum_j exp(s_j)
    (natural log); with ``return_probs`` also p [Hq, S, L + S].
    """
    S, Hq, D = q.shape
    Hkv = k_blk.shape[1]
    G = Hq // Hkv
    L = k_ctx.shape[0]
    K = np.concatenate([k_ctx, k_blk], axis=0)      # [L+S, Hkv, D]
    Vv = np.concatenate([v_ctx, v_blk], axis=0)
    # visible[i, j]: may block query i read key j of [context ; block]?
    visible = np.ones((S, L + S), dtype=bool)
    if causal_block:
        for i in range(S):
            visible[i, L + i + 1:] = False
    o = np.empty((S, Hq, D), dtype=np.float64)
    lse = np.empty((Hq, S), dtype=np.float64)
    probs = np.empty((Hq, S, K.shape[0]), dtype=np.float64) if return_probs else None
    for h in range(Hq):
        g = h // G
        s = sm_scale * (q[:, h, :] @ K[:, g, :].T)   # [S, L+S]
        if key_bias is not None:
            s = s + key_bias[None, :]
        s = np.where(visible, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        z = e.sum(axis=1, keepdims=True)
        p = e / z
        o[:, h, :] = p @ Vv[:, g, :]
        lse[h, :] = (m + np.log(z))[:, 0]
        if return_probs:
            probs[h] = p
    if return_probs:
        return o, lse, probs
    return o, lse


def denoise_attention(k_pool: np.ndarray, v_pool: np.ndarray, page_table: np.ndarray,
                      ctx_len: np.ndarray, page_size: int, q: np.ndarray, k_blk: np.ndarray,
                      v_blk: np.ndarray, sm_scale: float, dtype: str,
                      seqs: Optional[Sequence[int]] = None, causal_block: bool = False):
    """Batched two-segment attention over a paged context cache.

    Shapes as stored: pools [num_pages, Hkv, page_size, D]; page_table [B, max_pages];
    q [B, S, Hq, D]; k_blk, v_blk [B, S, Hkv, D].  ``seqs`` restricts the work to some
    sequences (the others are returned as NaN).  ``causal_block`` as in
    ``denoise_attention_seq``.  Returns o [B, S, Hq, D] and lse [B, Hq, S].
    """
    B, S, Hq, D = q.shape
    o = np.full((B, S, Hq, D), np.nan)
    lse = np.full((B, Hq, S), np.nan)
    for b in (range(B) if seqs is None else seqs):
        L = int(ctx_len[b])
        kc = decode(context_rows(k_pool, page_table[b], L, page_size), dtype)
        vc = decode(context_rows(v_pool, page_table[b], L, page_size), dtype)
        o[b], lse[b] = denoise_attention_seq(decode(q[b], dtype), kc, vc, decode(k_blk[b], dtype),
                                             decode(v_blk[b], dtype), sm_scale,
                                             causal_block=causal_block)
    return o, lse


# --------------------------------------------------------------------------- unmasking

@dataclasses.dataclass
class UnmaskResult:
    tokens: np.ndarray          # [S] int, updated
    masked: np.ndarray          # [S] bool, updated
    committed_now: np.ndarray   # [S] bool
    conf: np.ndarray            # [S] float64 (NaN where the position was already locked)
    argmax: np.ndarray          # [S] int (-1 where the position was already locked)
    fallback: bool              # the at-least-one rule chose the commit


def unmask_seq(logits: np.ndarray, masked: np.ndarray, tokens: np.ndarray, tau: float,
               step: int, T: int) -> UnmaskResult:
    """Confidence unmasking of one block at denoise step ``step`` (1-based) of ``T`` ([U]).

    For every still-masked position p (locked positions are skipped, their
    logits are never read):  m_p = max_v l_{p,v};  Z_p = sum_v exp(l_{p,v} - m_p);
    conf_p = 1 / Z_p (the largest softmax probability);  a_p = the lowest v with
    l_{p,v} = m_p.  Committed set C = {p masked : conf_p >= tau}; if C is empty and
    a position is still masked, C = {the most confident masked p} (lowest p on
    ties); at step T, C = every masked position.  Committed positions take token
    a_p and become unmasked; the others keep their token and stay masked.
    """
    S = masked.shape[0]
    masked = np.asarray(masked, dtype=bool)
    conf = np.full(S, np.nan)
    arg = np.full(S, -1, dtype=np.int64)
    for p in range(S):
        if not masked[p]:
            continue
        row = np.asarray(logits[p], dtype=np.float64)
        m = row.max()
        z = np.exp(row - m).sum()
        conf[p] = 1.0 / z
        arg[p] = int(np.argmax(row))            # first index of the maximum
    committed, fallback = commit_rule(conf, masked, tau, step, T)
    new_tokens = np.array(tokens, dtype=np.int64, copy=True)
    new_masked = masked.copy()
    for p in np.nonzero(committed)[0]:
        new_tokens[p] = arg[p]
        new_masked[p] = False
    return UnmaskResult(new_tokens, new_masked, committed, conf, arg, fallback)


def commit_rule(conf: np.ndarray, masked: np.ndarray, tau: float, step: int, T: int):
    """Which masked positions the step commits, given their confidences ([U]).

    C = {p masked : conf_p >= tau}; at step T (step >= T) C is every masked
    position; otherwise, if C is empty and a position is still masked, C holds
    the single most confident masked position (the lowest p on ties).  Only the
    entries of ``conf`` at masked positions are read.  Returns (committed [S]
    bool, fallback) where ``fallback`` says the at-least-one rule made the choice.
    """
    S = len(masked)
    masked = np.asarray(masked, dtype=bool)
    cand = [p for p in range(S) if masked[p]]
    chosen = [p for p in cand if conf[p] >= tau]
    fallback = False
    if step >= T:
        chosen = cand
    elif not chosen and cand:
        best = cand[0]
        for p in cand[1:]:
            if conf[p] > conf[best]:
                best = p
        chosen = [best]
        fallback = True
    committed = np.zeros(S, dtype=bool)
    committed[chosen] = True
    return committed, fallback


def unmask(logits: np.ndarray, masked: np.ndarray, tokens: np.ndarray, tau: float, step: int,
           T: int, dtype: str, seqs: Optional[Sequence[int]] = None):
    """Batched unmasking: logits [B, S, V] as stored; masked [B, S]; tokens [B, S].

    Returns a list of UnmaskResult (None for sequences outside ``seqs``)."""
    B = logits.shape[0]
    res = []
    for b in range(B):
        if seqs is not None and b not in seqs:
            res.append(None)
            continue
        rows = {}
        for p in range(logits.shape[1]):
            if masked[b, p]:
                rows[p] = decode(logits[b, p], dtype)
        # locked rows are passed as NaN placeholders: they must never be read
        lg = np.full((logits.shape[1], logits.shape[2]), np.nan)
        for p, r in rows.items():
            lg[p] = r
        res.append(unmask_seq(lg, masked[b], tokens[b], tau, step, T))
    return res


# --------------------------------------------------------------------------- commit / append

def kv_append(k_pool: np.ndarray, v_pool: np.ndarray, page_table: np.ndarray, ctx_len: np.ndarray,
              k_new: np.ndarray, v_new: np.ndarray, page_size: int,
              active: Optional[np.ndarray] = None) -> np.ndarray:
    """Commit a block into the context cache ([G]: the context tower extends its state).

    For every active sequence b and block position s < S, context position
    L_b + s receives the new key/value row (page ``page_table[b][(L_b+s)//page_size]``,
    slot ``(L_b+s) % page_size``); then L_b grows by S.  The pools are updated in
    place (as stored, no rounding); the new lengths are returned.
    """
    B, S = k_new.shape[:2]
    new_len = np.array(ctx_len, dtype=np.int64, copy=True)
    for b in range(B):
        if active is not None and not active[b]:
            continue
        L = int(ctx_len[b])
        if L + S > page_table.shape[1] * page_size:
            raise ValueError("block does not fit the sequence's pages")
        for s in range(S):
            j = L + s
            page = page_table[b, j // page_size]
            k_pool[page, :, j % page_size, :] = k_new[b, s]
            v_pool[page, :, j % page_size, :] = v_new[b, s]
        new_len[b] = L + S
    return new_len


# --------------------------------------------------------------------------- masked-diffusion loss

def linear_schedule_mask(u: np.ndarray, t: float) -> np.ndarray:
    """Corruption of a clean block at diffusion time t under the linear schedule ([T]).

    Each position is replaced by [MASK] with probability t and kept with
    probability 1 - t, independently of the others.  The uniform draws u_p in
    [0, 1) are inputs (one per position); position p is masked iff u_p < t, so
    P(masked) = t exactly.  t must lie in [0, 1].
    """
    if not 0.0 <= t <= 1.0:
        raise ValueError(f"diffusion time {t} outside [0, 1]")
    return np.asarray(u, dtype=np.float64) < t


def masked_nll_seq(logits: np.ndarray, targets: np.ndarray, masked: np.ndarray):
    """Negative log-likelihood of the clean tokens at the masked positions of one block ([T]).

    For every masked position p with clean token x_p:
        nll_p = log sum_v exp(l_{p,v}) - l_{p,x_p}      (= -log softmax(l_p)[x_p]),
    evaluated with the row maximum taken out first.  Unmasked positions are
    skipped (their logits are never read) and get NaN.  Returns nll [S], the sum
    over the masked positions and their count.
    """
    S = len(masked)
    nll = np.full(S, np.nan)
    total, count = 0.0, 0
    for p in range(S):
        if not masked[p]:
            continue
        row = np.asarray(logits[p], dtype=np.float64)
        m = row.max()
        lse = m + np.log(np.exp(row - m).sum())
        nll[p] = lse - row[int(targets[p])]
        total += nll[p]
        count += 1
    return nll, total, count


def masked_nll(logits: np.ndarray, targets: np.ndarray, masked: np.ndarray, dtype: str,
               seqs: Optional[Sequence[int]] = None):
    """Batched masked NLL: logits [B, S, V] as stored; targets, masked [B, S].

    Returns nll [B, S] (NaN where unmasked or outside ``seqs``), per-sequence sums
    [B] and counts [B] (NaN / -1 outside ``seqs``)."""
    B, S = masked.shape
    nll = np.full((B, S), np.nan)
    sums = np.full(B, np.nan)
    counts = np.full(B, -1, dtype=np.int64)
    for b in (range(B) if seqs is None else seqs):
        lg = np.full((S, logits.shape[2]), np.nan)
        for p in range(S):
            if masked[b, p]:
                lg[p] = decode(logits[b, p], dtype)
        nll[b], sums[b], counts[b] = masked_nll_seq(lg, targets[b], masked[b])
    return nll, sums, counts
