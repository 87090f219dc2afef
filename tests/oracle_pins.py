"""Checks that pin the float64 oracle to things other than itself.

Each ``check_*`` takes an implementation namespace ``impl`` exposing
``decode``, ``context_rows``, ``denoise_attention_seq``, ``denoise_attention``,
``unmask_seq``, ``commit_rule``, ``unmask``, ``kv_append``, ``linear_schedule_mask``,
``masked_nll_seq`` and ``masked_nll`` (the oracle, or a deliberately broken copy
of it) and raises AssertionError if the implementation disagrees
with:

* brute force (pure-Python loops, a different route to the same definition),
* a library routine in a case that reduces to it (PyTorch's float64
  ``scaled_dot_product_attention`` on a contiguous, unpaged key set; SciPy's
  ``softmax`` for the confidence),
* closed forms (equal keys give the mean of V; a dominant key returns its V row;
  a single spike of height a over V-1 zeros gives confidence e^a/(e^a+V-1)),
* invariants (convex combinations, -inf keys change nothing, physical page order
  is irrelevant, locked positions are never touched, every block finishes).

The decision rules being pinned are the sampling rule and the confidence trick of
the TwoTower summary (gist.science/de, "Training und Konditionierung — Sampling",
and "Der Konfidenz-Trick"), the attention visibility of its "Technisches
Resümee — Architektur" section, and the commit step of its
"Generierungsprozess" section.
"""
from __future__ import annotations

import math

import numpy as np
import scipy.special
import torch


# ------------------------------------------------------------------ helpers (no oracle code)

def _paged_from_contiguous(rng, ctx, page_size, extra_pages=2):
    """Scatter a contiguous [L, Hkv, D] context into a shuffled page pool; unused slots get NaN."""
    L, Hkv, D = ctx.shape
    n_own = max(1, -(-L // page_size))
    num_pages = n_own + extra_pages
    perm = rng.permutation(num_pages)
    table = perm[:n_own]
    pool = np.full((num_pages, Hkv, page_size, D), np.nan)
    for j in range(L):
        pool[table[j // page_size], :, j % page_size, :] = ctx[j]
    return pool, table


def _sdpa(q, K, V, scale, G):
    """PyTorch float64 SDPA. q [S,Hq,D]; K,V [N,Hkv,D] contiguous; KV heads repeated G times."""
    qt = torch.from_numpy(np.ascontiguousarray(q.transpose(1, 0, 2)))           # [Hq, S, D]
    kt = torch.from_numpy(np.ascontiguousarray(K.transpose(1, 0, 2))).repeat_interleave(G, 0)
    vt = torch.from_numpy(np.ascontiguousarray(V.transpose(1, 0, 2))).repeat_interleave(G, 0)
    o = torch.nn.functional.scaled_dot_product_attention(qt[None], kt[None], vt[None], scale=scale)
    return o[0].numpy().transpose(1, 0, 2)                                      # [S, Hq, D]


def _brute_attention(q, pool_k, pool_v, table, L, page_size, kb, vb, scale, causal_block=False):
    """Pure-Python attention: enumerate the visible keys by scanning the pages, weight each
    value by exp(score) and divide by the total weight (inputs are small, no overflow).
    With ``causal_block`` block query i skips the block keys after position i.
    Returns the outputs [S, Hq, D] and log(total weight) [Hq, S]."""
    S, Hq, D = q.shape
    Hkv = kb.shape[1]
    G = Hq // Hkv
    owner = {}
    for lp, page in enumerate(table):
        owner[int(page)] = lp
    keys = []                       # (k_row, v_row) per visible key, in any order
    for page in range(pool_k.shape[0]):
        if page not in owner:
            continue
        for slot in range(page_size):
            pos = owner[page] * page_size + slot
            if pos < L:
                keys.append((pool_k[page, :, slot, :], pool_v[page, :, slot, :]))
    out = np.zeros((S, Hq, D))
    lse = np.zeros((Hq, S))
    for i in range(S):
        seen = list(keys)
        for s in range(S):
            if causal_block and s > i:
                break
            seen.append((kb[s], vb[s]))
        for h in range(Hq):
            g = h // G
            w = []
            for kr, _ in seen:
                w.append(math.exp(scale * math.fsum(float(q[i, h, d]) * float(kr[g, d]) for d in range(D))))
            tot = math.fsum(w)
            lse[h, i] = math.log(tot)
            for d in range(D):
                out[i, h, d] = math.fsum(wj * float(vr[g, d]) for wj, (_, vr) in zip(w, seen)) / tot
    return out, lse


# ------------------------------------------------------------------ attention pins

def check_attention_bruteforce(impl, seed=0):
    rng = np.random.default_rng(seed)
    ps = 4
    for L in (0, 1, 3, 4, 5, 9):
        S, Hq, Hkv, D = 3, 4, 2, 3
        q = rng.normal(size=(S, Hq, D))
        ctx_k = rng.normal(size=(L, Hkv, D))
        ctx_v = rng.normal(size=(L, Hkv, D))
        kb, vb = rng.normal(size=(S, Hkv, D)), rng.normal(size=(S, Hkv, D))
        pk, table = _paged_from_contiguous(rng, ctx_k, ps)
        pv = np.full_like(pk, np.nan)
        for j in range(L):
            pv[table[j // ps], :, j % ps, :] = ctx_v[j]
        want, want_lse = _brute_attention(q, pk, pv, table, L, ps, kb, vb, 0.7)
        kc = impl.context_rows(pk, table, L, ps)
        vc = impl.context_rows(pv, table, L, ps)
        got, got_lse = impl.denoise_attention_seq(q, kc, vc, kb, vb, 0.7)
        assert np.allclose(got, want, rtol=0, atol=1e-12), (L, np.abs(got - want).max())
        assert np.allclose(got_lse, want_lse, rtol=0, atol=1e-12), (L, np.abs(got_lse - want_lse).max())


def check_attention_sdpa(impl, seed=1):
    """Against PyTorch's SDPA on the contiguous concatenation [context ; block] (L = 0 is the
    plain bidirectional in-block attention)."""
    rng = np.random.default_rng(seed)
    for L, ps, (S, Hq, Hkv, D) in ((0, 8, (16, 8, 2, 16)), (37, 8, (16, 8, 2, 16)),
                                   (64, 16, (16, 4, 1, 32)), (5, 4, (2, 6, 3, 5))):
        q = rng.normal(size=(S, Hq, D))
        ctx_k, ctx_v = rng.normal(size=(L, Hkv, D)), rng.normal(size=(L, Hkv, D))
        kb, vb = rng.normal(size=(S, Hkv, D)), rng.normal(size=(S, Hkv, D))
        scale = 1.0 / math.sqrt(D)
        want = _sdpa(q, np.concatenate([ctx_k, kb]), np.concatenate([ctx_v, vb]), scale, Hq // Hkv)
        pk, table = _paged_from_contiguous(rng, ctx_k, ps)
        pv = np.full_like(pk, np.nan)
        for j in range(L):
            pv[table[j // ps], :, j % ps, :] = ctx_v[j]
        got, _ = impl.denoise_attention_seq(q, impl.context_rows(pk, table, L, ps),
                                            impl.context_rows(pv, table, L, ps), kb, vb, scale)
        assert np.allclose(got, want, rtol=0, atol=1e-12), (L, np.abs(got - want).max())


def check_attention_closed_forms(impl, seed=2):
    rng = np.random.default_rng(seed)
    S, Hq, Hkv, D, L = 4, 4, 2, 8, 11
    q = rng.normal(size=(S, Hq, D))
    # (1) all keys equal -> uniform weights -> the mean of V over the L+S keys; lse = c + log(L+S)
    k_all = rng.normal(size=(Hkv, D))
    kc = np.broadcast_to(k_all, (L, Hkv, D)).copy()
    kb = np.broadcast_to(k_all, (S, Hkv, D)).copy()
    vc, vb = rng.normal(size=(L, Hkv, D)), rng.normal(size=(S, Hkv, D))
    o, lse = impl.denoise_attention_seq(q, kc, vc, kb, vb, 0.5)
    mean_v = np.concatenate([vc, vb]).mean(axis=0)            # [Hkv, D]
    G = Hq // Hkv
    for h in range(Hq):
        assert np.allclose(o[:, h, :], mean_v[h // G][None, :], rtol=0, atol=1e-12)
        c = 0.5 * (q[:, h, :] @ k_all[h // G])
        assert np.allclose(lse[h], c + math.log(L + S), rtol=0, atol=1e-12)
    # (2) one context key scores 60 above every other key for head 0 -> its V row.
    # Every other key is tiny (|score| < 0.1), so the planted key carries all but
    # about (L+S) * e^-59.9 of the weight.
    kc = rng.normal(size=(L, Hkv, D)) * 1e-3
    kb = rng.normal(size=(S, Hkv, D)) * 1e-3
    jstar = 7
    u = rng.normal(size=D)
    u /= np.linalg.norm(u)
    q2 = q.copy()
    q2[:, 0, :] = 10.0 * u
    kc[jstar, 0, :] = 6.0 * u
    o, _ = impl.denoise_attention_seq(q2, kc, vc, kb, vb, 1.0)
    assert np.allclose(o[:, 0, :], vc[jstar, 0, :][None, :], rtol=0, atol=1e-15)
    # the same key for head G (KV head 1) does not dominate: KV heads are not mixed
    assert not np.allclose(o[:, G, :], vc[jstar, 1 % Hkv, :][None, :], rtol=0, atol=1e-3)


def check_attention_invariants(impl, seed=3):
    rng = np.random.default_rng(seed)
    S, Hq, Hkv, D, L = 5, 6, 3, 4, 13
    q = rng.normal(size=(S, Hq, D)) * 2
    kc, vc = rng.normal(size=(L, Hkv, D)), rng.normal(size=(L, Hkv, D))
    kb, vb = rng.normal(size=(S, Hkv, D)), rng.normal(size=(S, Hkv, D))
    o, lse, p = impl.denoise_attention_seq(q, kc, vc, kb, vb, 0.9, return_probs=True)
    # convex combinations of V: weights >= 0 summing to 1, outputs inside the hull per coordinate
    assert (p >= 0).all() and np.allclose(p.sum(axis=-1), 1.0, rtol=0, atol=1e-13)
    allv = np.concatenate([vc, vb])
    G = Hq // Hkv
    for h in range(Hq):
        lo, hi = allv[:, h // G].min(axis=0), allv[:, h // G].max(axis=0)
        assert (o[:, h] >= lo - 1e-12).all() and (o[:, h] <= hi + 1e-12).all()
    # an extra context key whose score is -inf changes nothing
    kx = np.concatenate([kc, rng.normal(size=(1, Hkv, D))])
    vx = np.concatenate([vc, rng.normal(size=(1, Hkv, D)) * 1e6])
    bias = np.zeros(L + 1 + S)
    bias[L] = -np.inf
    o2, lse2 = impl.denoise_attention_seq(q, kx, vx, kb, vb, 0.9, key_bias=bias)
    assert np.allclose(o2, o, rtol=0, atol=1e-14) and np.allclose(lse2, lse, rtol=0, atol=1e-14)
    # permuting the context positions (keys with their values) changes nothing: no positional logic
    perm = rng.permutation(L)
    o3, _ = impl.denoise_attention_seq(q, kc[perm], vc[perm], kb, vb, 0.9)
    assert np.allclose(o3, o, rtol=0, atol=1e-13)
    # the block's own keys are all visible to every block query (bidirectional): the last block
    # position's key/value influences the first block query
    vb2 = vb.copy()
    vb2[-1] += 5.0
    o4, _ = impl.denoise_attention_seq(q, kc, vc, kb, vb2, 0.9)
    assert (np.abs(o4[0] - o[0]) > 1e-6).all()
    # physical page order is irrelevant, and slots past L are never read
    ps = 4
    pk, table = _paged_from_contiguous(rng, kc, ps, extra_pages=3)
    pv = np.full_like(pk, np.nan)
    for j in range(L):
        pv[table[j // ps], :, j % ps, :] = vc[j]
    o5, _ = impl.denoise_attention_seq(q, impl.context_rows(pk, table, L, ps),
                                       impl.context_rows(pv, table, L, ps), kb, vb, 0.9)
    assert np.array_equal(o5, o)


def check_attention_segment_merge(impl, seed=14):
    """Attention over [context ; block] is the log-sum-exp weighted merge of attention over
    each segment alone (the block removed with -inf scores, or no context):
    lse = logaddexp(lse_c, lse_b) and o = (e^lse_c o_c + e^lse_b o_b) / e^lse."""
    rng = np.random.default_rng(seed)
    S, Hq, Hkv, D, L = 4, 6, 2, 5, 19
    q = rng.normal(size=(S, Hq, D)) * 1.5
    kc, vc = rng.normal(size=(L, Hkv, D)), rng.normal(size=(L, Hkv, D))
    kb, vb = rng.normal(size=(S, Hkv, D)), rng.normal(size=(S, Hkv, D))
    o, lse = impl.denoise_attention_seq(q, kc, vc, kb, vb, 0.8)
    bias = np.zeros(L + S)
    bias[L:] = -np.inf
    o_c, lse_c = impl.denoise_attention_seq(q, kc, vc, kb, vb, 0.8, key_bias=bias)
    empty = np.zeros((0, Hkv, D))
    o_b, lse_b = impl.denoise_attention_seq(q, empty, empty, kb, vb, 0.8)
    want_lse = np.logaddexp(lse_c, lse_b)                      # [Hq, S]
    assert np.allclose(lse, want_lse, rtol=0, atol=1e-12)
    w_c = np.exp(lse_c - want_lse).T[:, :, None]               # [S, Hq, 1]
    w_b = np.exp(lse_b - want_lse).T[:, :, None]
    assert np.allclose(o, w_c * o_c + w_b * o_b, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ causal-block attention pins
# The context tower taking in a committed block: block query i sees every context key and
# the block keys 0..i (gist.science summary, "Technisches Resümee — Architektur": the frozen
# tower is causal over the prompt and the committed tokens).

def check_causal_block_bruteforce(impl, seed=7):
    rng = np.random.default_rng(seed)
    ps = 4
    for L in (0, 1, 3, 5, 9):
        S, Hq, Hkv, D = 4, 4, 2, 3
        q = rng.normal(size=(S, Hq, D))
        ctx_k, ctx_v = rng.normal(size=(L, Hkv, D)), rng.normal(size=(L, Hkv, D))
        kb, vb = rng.normal(size=(S, Hkv, D)), rng.normal(size=(S, Hkv, D))
        pk, table = _paged_from_contiguous(rng, ctx_k, ps)
        pv = np.full_like(pk, np.nan)
        for j in range(L):
            pv[table[j // ps], :, j % ps, :] = ctx_v[j]
        want, want_lse = _brute_attention(q, pk, pv, table, L, ps, kb, vb, 0.8, causal_block=True)
        got, got_lse = impl.denoise_attention_seq(q, impl.context_rows(pk, table, L, ps),
                                                  impl.context_rows(pv, table, L, ps), kb, vb, 0.8,
                                                  causal_block=True)
        assert np.allclose(got, want, rtol=0, atol=1e-12), (L, np.abs(got - want).max())
        assert np.allclose(got_lse, want_lse, rtol=0, atol=1e-12), (L, np.abs(got_lse - want_lse).max())


def check_causal_block_sdpa(impl, seed=8):
    """With no context the view is PyTorch's causal SDPA (is_causal=True); with a context,
    block query i is plain SDPA of that one query over [context ; block keys 0..i]."""
    rng = np.random.default_rng(seed)
    S, Hq, Hkv, D = 16, 8, 2, 16
    scale = 1.0 / math.sqrt(D)
    G = Hq // Hkv
    q = rng.normal(size=(S, Hq, D))
    kb, vb = rng.normal(size=(S, Hkv, D)), rng.normal(size=(S, Hkv, D))
    empty = np.zeros((0, Hkv, D))
    got, _ = impl.denoise_attention_seq(q, empty, empty, kb, vb, scale, causal_block=True)
    qt = torch.from_numpy(np.ascontiguousarray(q.transpose(1, 0, 2)))
    kt = torch.from_numpy(np.ascontiguousarray(kb.transpose(1, 0, 2))).repeat_interleave(G, 0)
    vt = torch.from_numpy(np.ascontiguousarray(vb.transpose(1, 0, 2))).repeat_interleave(G, 0)
    want = torch.nn.functional.scaled_dot_product_attention(qt[None], kt[None], vt[None], scale=scale,
                                                            is_causal=True)[0].numpy().transpose(1, 0, 2)
    assert np.allclose(got, want, rtol=0, atol=1e-12), np.abs(got - want).max()
    for L in (1, 21, 64):
        ctx_k, ctx_v = rng.normal(size=(L, Hkv, D)), rng.normal(size=(L, Hkv, D))
        got, _ = impl.denoise_attention_seq(q, ctx_k, ctx_v, kb, vb, scale, causal_block=True)
        for i in range(S):
            want_i = _sdpa(q[i:i + 1], np.concatenate([ctx_k, kb[:i + 1]]),
                           np.concatenate([ctx_v, vb[:i + 1]]), scale, G)
            assert np.allclose(got[i:i + 1], want_i, rtol=0, atol=1e-12), (L, i)


def check_causal_block_closed_forms(impl, seed=9):
    rng = np.random.default_rng(seed)
    S, Hq, Hkv, D = 5, 4, 2, 6
    G = Hq // Hkv
    q = rng.normal(size=(S, Hq, D))
    vb = rng.normal(size=(S, Hkv, D))
    kb = rng.normal(size=(S, Hkv, D))
    empty = np.zeros((0, Hkv, D))
    # (1) no context: block query 0 sees only block key 0 -> exactly its V row, lse = its score
    o, lse = impl.denoise_attention_seq(q, empty, empty, kb, vb, 0.6, causal_block=True)
    for h in range(Hq):
        assert np.array_equal(o[0, h], vb[0, h // G])
        assert math.isclose(lse[h, 0], 0.6 * float(q[0, h] @ kb[0, h // G]), rel_tol=0, abs_tol=1e-13)
    # (2) all keys equal -> block query i averages V over the L + i + 1 keys it sees
    L = 7
    k_all = rng.normal(size=(Hkv, D))
    kc = np.broadcast_to(k_all, (L, Hkv, D)).copy()
    kbe = np.broadcast_to(k_all, (S, Hkv, D)).copy()
    vc = rng.normal(size=(L, Hkv, D))
    o, lse = impl.denoise_attention_seq(q, kc, vc, kbe, vb, 0.6, causal_block=True)
    allv = np.concatenate([vc, vb])
    for i in range(S):
        mean_v = allv[:L + i + 1].mean(axis=0)
        for h in range(Hq):
            assert np.allclose(o[i, h], mean_v[h // G], rtol=0, atol=1e-12), (i, h)
            c = 0.6 * float(q[i, h] @ k_all[h // G])
            assert math.isclose(lse[h, i], c + math.log(L + i + 1), rel_tol=0, abs_tol=1e-12)


def check_causal_block_invariants(impl, seed=10):
    rng = np.random.default_rng(seed)
    S, Hq, Hkv, D, L = 6, 4, 1, 5, 9
    q = rng.normal(size=(S, Hq, D))
    kc, vc = rng.normal(size=(L, Hkv, D)), rng.normal(size=(L, Hkv, D))
    kb, vb = rng.normal(size=(S, Hkv, D)), rng.normal(size=(S, Hkv, D))
    o, lse = impl.denoise_attention_seq(q, kc, vc, kb, vb, 0.7, causal_block=True)
    ob, lseb = impl.denoise_attention_seq(q, kc, vc, kb, vb, 0.7)
    # the last block position sees everything: same as the bidirectional view
    assert np.allclose(o[-1], ob[-1], rtol=0, atol=1e-14) and np.allclose(lse[:, -1], lseb[:, -1], rtol=0,
                                                                           atol=1e-14)
    # earlier positions do not (the later block keys carry weight in the bidirectional view)
    assert (np.abs(o[:-1] - ob[:-1]).max(axis=(1, 2)) > 1e-6).all()
    # a later block key or value never reaches an earlier query: bitwise unchanged rows
    for j in range(S):
        kb2, vb2 = kb.copy(), vb.copy()
        kb2[j] += 3.0
        vb2[j] -= 7.0
        o2, lse2 = impl.denoise_attention_seq(q, kc, vc, kb2, vb2, 0.7, causal_block=True)
        assert np.array_equal(o2[:j], o[:j]) and np.array_equal(lse2[:, :j], lse[:, :j]), j
        assert (np.abs(o2[j:] - o[j:]).max(axis=(1, 2)) > 1e-6).all(), j
    # a block query that sees its own key dominate returns that key's V row
    u = rng.normal(size=D)
    u /= np.linalg.norm(u)
    q3, kb3 = q * 1e-3, kb * 1e-3
    kc3 = kc * 1e-3
    i = 3
    q3[i, 0] = 10.0 * u
    kb3[i, 0] = 6.0 * u
    o3, _ = impl.denoise_attention_seq(q3, kc3, vc, kb3, vb, 1.0, causal_block=True)
    assert np.allclose(o3[i, 0], vb[i, 0], rtol=0, atol=1e-15)


# ------------------------------------------------------------------ unmasking pins

def _brute_conf(row):
    m = max(row)
    z = math.fsum(math.exp(x - m) for x in row)
    arg = min(i for i, x in enumerate(row) if x == m)
    return 1.0 / z, arg


def check_unmask_closed_forms(impl):
    V, tau = 1024, 0.9
    # spike of height a at token k over zeros: conf = e^a / (e^a + V - 1)
    def spike_height(conf):
        return math.log(conf * (V - 1) / (1.0 - conf))
    rows, want_conf = [], []
    for k, c in ((5, tau + 1e-3), (900, tau - 1e-3), (0, 0.5), (1023, 0.99)):
        a = spike_height(c)
        r = np.zeros(V)
        r[k] = a
        rows.append(r)
        want_conf.append(math.exp(a) / (math.exp(a) + V - 1))
    # all logits equal: conf = 1/V, argmax = 0
    rows.append(np.full(V, 3.25))
    want_conf.append(1.0 / V)
    # two tied maxima: the lower token id wins
    r = np.zeros(V)
    r[17] = r[400] = 9.0
    rows.append(r)
    want_conf.append(math.exp(9.0) / (2 * math.exp(9.0) + V - 2))
    lg = np.stack(rows)
    S = lg.shape[0]
    res = impl.unmask_seq(lg, np.ones(S, bool), np.full(S, -7), tau, 1, 8)
    assert np.allclose(res.conf, want_conf, rtol=1e-13, atol=0)
    assert list(res.argmax) == [5, 900, 0, 1023, 0, 17]
    assert list(res.committed_now) == [True, False, False, True, False, False]
    assert list(res.tokens) == [5, -7, -7, 1023, -7, -7]
    assert not res.fallback


def check_unmask_bruteforce(impl, seed=4):
    rng = np.random.default_rng(seed)
    for trial in range(6):
        S, V = 6, 50
        lg = rng.normal(scale=3.0, size=(S, V))
        lg[np.arange(S), rng.integers(0, V, S)] += rng.uniform(0, 12, S)
        lg = np.round(lg * 4) / 4          # coarse grid: exact ties happen
        masked = rng.random(S) < 0.7
        masked[0] = True
        tau = [0.9, 0.3, 0.05, 0.6, 0.999, 0.2][trial]
        res = impl.unmask_seq(lg, masked, np.arange(S) + 100, tau, 1, 4)
        conf, arg = {}, {}
        for p in range(S):
            if masked[p]:
                conf[p], arg[p] = _brute_conf([float(x) for x in lg[p]])
                assert abs(res.conf[p] - conf[p]) <= 1e-14 and res.argmax[p] == arg[p]
                sm = scipy.special.softmax(lg[p]).max()
                assert abs(res.conf[p] - sm) <= 1e-13
        chosen = [p for p in conf if conf[p] >= tau]
        if not chosen:
            best = max(conf.values())
            chosen = [min(p for p in conf if conf[p] == best)]
        for p in range(S):
            want_commit = p in chosen
            assert res.committed_now[p] == want_commit
            assert res.masked[p] == (masked[p] and not want_commit)
            assert res.tokens[p] == (arg[p] if want_commit else p + 100)


def check_unmask_rules(impl):
    V = 64
    base = np.zeros((4, V))
    # conf < tau everywhere; rows 1 and 2 identical (tie) and most confident -> fallback picks row 1
    base[0, 3] = 1.0
    base[1, 9] = 2.0
    base[2, 9] = 2.0
    base[3, 5] = 0.5
    res = impl.unmask_seq(base, np.ones(4, bool), np.full(4, -1), 0.9, 1, 4)
    assert res.fallback and list(res.committed_now) == [False, True, False, False]
    assert res.tokens[1] == 9 and res.masked.sum() == 3
    # at step T every still-masked position is committed, whatever its confidence
    res = impl.unmask_seq(base, np.array([True, False, True, True]), np.array([-1, 42, -1, -1]),
                          0.9, 4, 4)
    assert list(res.committed_now) == [True, False, True, True] and not res.masked.any()
    assert list(res.tokens) == [3, 42, 9, 5]
    # locked positions are never read (NaN logits there) and never change
    lg = base.copy()
    lg[1] = np.nan
    res = impl.unmask_seq(lg, np.array([True, False, True, True]), np.array([-1, 42, -1, -1]),
                          0.9, 1, 4)
    assert res.tokens[1] == 42 and not res.committed_now[1] and np.isnan(res.conf[1])
    assert np.isfinite(res.conf[[0, 2, 3]]).all()
    # several confident positions: exactly the set {conf >= tau} (adaptive count), no fallback
    lg = np.zeros((5, V))
    for p, a in enumerate((20.0, 1.0, 30.0, 15.0, 0.0)):
        lg[p, p] = a
    res = impl.unmask_seq(lg, np.ones(5, bool), np.full(5, -1), 0.9, 1, 4)
    want = [math.exp(a) / (math.exp(a) + V - 1) >= 0.9 for a in (20.0, 1.0, 30.0, 15.0, 0.0)]
    assert list(res.committed_now) == want and not res.fallback
    # nothing masked: nothing happens
    res = impl.unmask_seq(lg, np.zeros(5, bool), np.arange(5), 0.9, 2, 4)
    assert not res.committed_now.any() and list(res.tokens) == list(range(5))


def check_block_loop(impl, seed=5):
    """Every block finishes within T steps, each step commits at least one position and a
    committed token never changes afterwards."""
    rng = np.random.default_rng(seed)
    S, V, T = 16, 256, 6
    for blk in range(5):
        masked = np.ones(S, bool)
        tokens = np.full(S, -1)
        history = {}
        for step in range(1, T + 1):
            lg = rng.normal(scale=3.0, size=(S, V))
            lg[np.arange(S), rng.integers(0, V, S)] += rng.uniform(0, 12, S)
            before = masked.sum()
            res = impl.unmask_seq(lg, masked, tokens, 0.9, step, T)
            assert res.committed_now.sum() >= 1 and res.masked.sum() == before - res.committed_now.sum()
            for p, t in history.items():
                assert res.tokens[p] == t
            for p in np.nonzero(res.committed_now)[0]:
                history[int(p)] = int(res.tokens[p])
            masked, tokens = res.masked, res.tokens
            if not masked.any():
                break
        assert not masked.any()


# ------------------------------------------------------------------ append pins

def check_append(impl, seed=6):
    rng = np.random.default_rng(seed)
    ps, Hkv, D, S, B = 4, 2, 3, 5, 3
    lens = np.array([0, 6, 8])
    maxp = 4
    num_pages = B * maxp + 1
    perm = rng.permutation(num_pages)
    table = perm[: B * maxp].reshape(B, maxp)
    ctx = [rng.normal(size=(L, Hkv, D)) for L in lens]
    kp = np.full((num_pages, Hkv, ps, D), np.nan)
    vp = np.full((num_pages, Hkv, ps, D), np.nan)
    vctx = [rng.normal(size=(L, Hkv, D)) for L in lens]
    for b in range(B):
        for j in range(lens[b]):
            kp[table[b, j // ps], :, j % ps] = ctx[b][j]
            vp[table[b, j // ps], :, j % ps] = vctx[b][j]
    kn, vn = rng.normal(size=(B, S, Hkv, D)), rng.normal(size=(B, S, Hkv, D))
    active = np.array([True, True, False])
    kp0, vp0 = kp.copy(), vp.copy()
    new_len = impl.kv_append(kp, vp, table, lens, kn, vn, ps, active=active)
    assert list(new_len) == [5, 11, 8]
    for b in range(B):
        got_k = impl.context_rows(kp, table[b], int(new_len[b]), ps)
        want_k = np.concatenate([ctx[b], kn[b]]) if active[b] else ctx[b]
        assert np.array_equal(got_k, want_k)
    # inactive sequence and foreign pages untouched (NaN-aware equality)
    own = set(table[0]) | set(table[1])
    for page in range(num_pages):
        if page not in own:
            assert np.array_equal(kp[page], kp0[page], equal_nan=True)
    # attention after the append equals SDPA over the contiguous concatenation
    q = rng.normal(size=(S, 2 * Hkv, D))
    kb, vb = rng.normal(size=(S, Hkv, D)), rng.normal(size=(S, Hkv, D))
    b = 1
    o, _ = impl.denoise_attention_seq(q, impl.context_rows(kp, table[b], 11, ps),
                                      impl.context_rows(vp, table[b], 11, ps), kb, vb, 0.6)
    want = _sdpa(q, np.concatenate([ctx[b], kn[b], kb]), np.concatenate([vctx[b], vn[b], vb]), 0.6, 2)
    assert np.allclose(o, want, rtol=0, atol=1e-12)
    # a block that does not fit the sequence's pages is refused
    try:
        impl.kv_append(kp, vp, table, np.array([14, 0, 0]), kn, vn, ps)
    except ValueError:
        pass
    else:
        raise AssertionError("capacity overflow not detected")


# ------------------------------------------------------------------ masked-diffusion loss pins
# Training side (gist.science summary, "Training und Konditionierung — Maskierte Diffusion"):
# clean blocks masked on a linear schedule; NLL of the clean tokens at the masked positions.

def check_linear_schedule(impl, seed=11):
    rng = np.random.default_rng(seed)
    u = rng.random(200_000)
    assert not impl.linear_schedule_mask(u, 0.0).any()
    assert impl.linear_schedule_mask(u, 1.0).all()
    prev = None
    for t in (0.05, 0.3, 0.5, 0.9):
        m = impl.linear_schedule_mask(u, t)
        # P(masked) = t: the fraction is binomial, within 5 standard deviations of t
        sd = math.sqrt(t * (1 - t) / u.size)
        assert abs(m.mean() - t) < 5 * sd, (t, m.mean())
        if prev is not None:
            assert (m | ~prev).all()             # a later time masks a superset
        prev = m
    try:
        impl.linear_schedule_mask(u[:4], 1.5)
    except ValueError:
        pass
    else:
        raise AssertionError("a time outside [0, 1] was accepted")


def check_masked_nll_closed_forms(impl):
    V, S = 1000, 4
    # all logits equal: every token has probability 1/V -> nll = log V
    nll, tot, cnt = impl.masked_nll_seq(np.full((S, V), 2.5), np.array([0, 7, 999, 3]), np.ones(S, bool))
    assert np.allclose(nll, math.log(V), rtol=0, atol=1e-12) and cnt == S
    assert math.isclose(tot, S * math.log(V), rel_tol=1e-14)
    # one spike of height a over zeros: at the target nll = log(e^a + V - 1) - a, elsewhere log(e^a + V - 1)
    a = 7.0
    lg = np.zeros((S, V))
    lg[:, 5] = a
    tg = np.array([5, 6, 5, 0])
    nll, _, _ = impl.masked_nll_seq(lg, tg, np.ones(S, bool))
    z = math.log(math.exp(a) + V - 1)
    assert np.allclose(nll, [z - a, z, z - a, z], rtol=0, atol=1e-12)
    # unmasked rows are never read (NaN there) and do not count
    lg[1] = np.nan
    lg[3] = np.nan
    nll, tot, cnt = impl.masked_nll_seq(lg, tg, np.array([True, False, True, False]))
    assert cnt == 2 and math.isclose(tot, 2 * (z - a), rel_tol=1e-13)
    assert np.isnan(nll[1]) and np.isnan(nll[3])


def check_masked_nll_library(impl, seed=12):
    """Against PyTorch's float64 cross entropy on the masked rows."""
    rng = np.random.default_rng(seed)
    S, V = 16, 300
    lg = rng.normal(0, 3, size=(S, V))
    tg = rng.integers(0, V, size=S)
    mk = rng.random(S) < 0.6
    nll, tot, cnt = impl.masked_nll_seq(lg, tg, mk)
    want = torch.nn.functional.cross_entropy(torch.from_numpy(lg[mk]), torch.from_numpy(tg[mk]),
                                             reduction="none").numpy()
    assert np.allclose(nll[mk], want, rtol=0, atol=1e-12)
    assert cnt == int(mk.sum()) and math.isclose(tot, float(want.sum()), rel_tol=1e-13)


def check_masked_nll_invariants(impl, seed=13):
    rng = np.random.default_rng(seed)
    S, V = 5, 64
    lg = rng.normal(0, 2, size=(S, V))
    tg = rng.integers(0, V, size=S)
    mk = np.ones(S, bool)
    nll, _, _ = impl.masked_nll_seq(lg, tg, mk)
    assert (nll >= 0).all()
    # a constant added to a row changes nothing; very large logits stay finite (the maximum is taken out)
    nll2, _, _ = impl.masked_nll_seq(lg + 1e4, tg, mk)
    assert np.allclose(nll2, nll, rtol=0, atol=1e-9)
    nll3, _, _ = impl.masked_nll_seq(lg * 200.0, tg, mk)
    assert np.isfinite(nll3).all()
    # exp(-nll) over every possible clean token of a row sums to 1 (a probability distribution)
    for p in range(S):
        probs = [math.exp(-impl.masked_nll_seq(lg[p:p + 1], np.array([v]), np.ones(1, bool))[0][0])
                 for v in range(V)]
        assert math.isclose(math.fsum(probs), 1.0, rel_tol=0, abs_tol=1e-13)
    # brute force with math.fsum on the unshifted values (moderate logits, no overflow)
    for p in range(S):
        want = math.log(math.fsum(math.exp(float(x)) for x in lg[p])) - float(lg[p, tg[p]])
        assert math.isclose(nll[p], want, rel_tol=0, abs_tol=1e-12)


# ------------------------------------------------------------------ decoding and the batched wrappers

def _torch_decode_bf16(bits):
    """bf16 bit patterns -> float64 through PyTorch's own bfloat16 conversion (no oracle code)."""
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.double().numpy()


def check_decode(impl, seed=15):
    """Every one of the 65536 bf16 bit patterns decodes to the value PyTorch gives it (NaN
    patterns to NaN), and float32 storage decodes to its exact float64 value."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):          # signalling-NaN patterns widen with a warning
        got = impl.decode(bits, "bf16")
    want = _torch_decode_bf16(bits)
    nan = np.isnan(want)
    assert nan.sum() == 254                       # 2 signs x 127 non-zero mantissas at exponent 255
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))   # -0.0 stays negative
    # a few values written out from the bfloat16 format: sign, 8 exponent bits, 7 mantissa bits
    spot = {0x3F80: 1.0, 0xBF80: -1.0, 0x4049: 3.140625, 0x0001: 2.0 ** -133, 0x7F7F: (2 - 2 ** -7) * 2.0 ** 127,
            0x7F80: math.inf, 0xFF80: -math.inf, 0x3C00: 2.0 ** -7, 0xC2F7: -123.5}
    for b, v in spot.items():
        assert impl.decode(np.array([b], np.uint16), "bf16")[0] == v, hex(b)
    # shape is kept
    with np.errstate(invalid="ignore"):
        assert impl.decode(bits.reshape(256, 256), "bf16").shape == (256, 256)
    # float32 storage: exact widening, specials included
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(1000).astype(np.float32) * np.float32(1e3)
    x[:6] = [0.0, -0.0, np.inf, -np.inf, np.float32(1e-45), np.float32(3.4e38)]
    got = impl.decode(x, "f32")
    assert got.dtype == np.float64
    assert np.array_equal(got, torch.from_numpy(x).double().numpy())
    assert np.signbit(got[1])


def check_commit_rule(impl):
    """The commit rule on confidences written out by hand."""
    nan = float("nan")
    cases = [
        # conf, masked, tau, step, T -> committed, fallback
        ([0.95, 0.2, 0.9, 0.5], [1, 1, 1, 1], 0.9, 1, 4, [1, 0, 1, 0], False),   # >= tau, tau itself commits
        ([0.3, 0.7, 0.7, 0.1], [1, 1, 1, 1], 0.9, 2, 4, [0, 1, 0, 0], True),     # fallback, tie -> lowest p
        ([0.3, 0.7, 0.8, 0.1], [1, 1, 1, 1], 0.9, 2, 4, [0, 0, 1, 0], True),     # fallback, most confident
        ([0.3, nan, 0.2, 0.1], [1, 0, 1, 1], 0.9, 3, 4, [1, 0, 0, 0], True),     # locked entries not read
        ([0.3, nan, 0.2, 0.1], [1, 0, 1, 1], 0.9, 4, 4, [1, 0, 1, 1], False),    # step T: all masked
        ([0.3, nan, 0.2, 0.1], [1, 0, 1, 1], 0.9, 7, 4, [1, 0, 1, 1], False),    # past T as well
        ([0.99, 0.99, 0.99], [0, 0, 0], 0.9, 1, 4, [0, 0, 0], False),            # nothing masked
        ([0.99, 0.95, 0.2], [0, 1, 1], 0.9, 1, 4, [0, 1, 0], False),             # locked confident row ignored
        ([0.5], [1], 0.5, 1, 4, [1], False),                                     # exactly tau
        ([0.5], [1], 0.5000001, 1, 4, [1], True),                                # just above: fallback
    ]
    for conf, masked, tau, step, T, want, fb in cases:
        com, fallback = impl.commit_rule(np.array(conf), np.array(masked, bool), tau, step, T)
        assert [int(c) for c in com] == want, (conf, masked, tau, step, T)
        assert bool(fallback) == fb, (conf, masked, tau, step, T)


def _walk_pages(pool, table_row, L, page_size):
    """The first L context rows of a sequence by an explicit loop over positions."""
    rows = []
    for j in range(L):
        rows.append(pool[int(table_row[j // page_size]), :, j % page_size, :])
    return np.stack(rows) if rows else np.zeros((0, pool.shape[1], pool.shape[3]), pool.dtype)


def check_batched_wrappers(impl, seed=16):
    """The batched entry points equal a loop over the per-sequence functions on a ragged
    three-sequence batch: pages walked position by position, values decoded by PyTorch,
    locked rows given as NaN (they must not be read), and the ``seqs`` selection honoured."""
    rng = np.random.default_rng(seed)
    B, S, Hq, Hkv, D, page, V = 3, 4, 4, 2, 8, 4, 50
    lens = np.array([5, 0, 11])
    maxp = 3
    num_pages = B * maxp + 2
    table = rng.permutation(num_pages)[:B * maxp].reshape(B, maxp)
    f32 = lambda shape: rng.standard_normal(shape).astype(np.float32)   # noqa: E731
    bits = lambda x: (x.view(np.uint32) >> 16).astype(np.uint16)         # noqa: E731  (truncation: exact bf16 values)
    kp, vp = bits(f32((num_pages, Hkv, page, D))), bits(f32((num_pages, Hkv, page, D)))
    q, kb, vb = bits(f32((B, S, Hq, D))), bits(f32((B, S, Hkv, D))), bits(f32((B, S, Hkv, D)))
    dec = _torch_decode_bf16
    o, lse = impl.denoise_attention(kp, vp, table, lens, page, q, kb, vb, 0.3, "bf16")
    for b in range(B):
        kc = dec(_walk_pages(kp, table[b], int(lens[b]), page))
        vc = dec(_walk_pages(vp, table[b], int(lens[b]), page))
        wo, wl = impl.denoise_attention_seq(dec(q[b]), kc, vc, dec(kb[b]), dec(vb[b]), 0.3)
        assert np.array_equal(o[b], wo) and np.array_equal(lse[b], wl), b
    o2, lse2 = impl.denoise_attention(kp, vp, table, lens, page, q, kb, vb, 0.3, "bf16", seqs=[2])
    assert np.isnan(o2[:2]).all() and np.isnan(lse2[:2]).all() and np.array_equal(o2[2], o[2])
    # unmasking: locked rows are passed as NaN to the per-sequence rule
    lg = bits(f32((B, S, V)) * np.float32(3))
    masked = np.array([[1, 0, 1, 1], [0, 0, 0, 0], [1, 1, 0, 1]], np.uint8)
    tokens = np.where(masked == 1, -1, 7 + np.arange(B * S).reshape(B, S))
    res = impl.unmask(lg, masked, tokens, 0.9, 2, 4, "bf16")
    for b in range(B):
        rows = np.full((S, V), np.nan)
        for p in range(S):
            if masked[b, p]:
                rows[p] = dec(lg[b, p])
        want = impl.unmask_seq(rows, masked[b].astype(bool), tokens[b], 0.9, 2, 4)
        got = res[b]
        assert np.array_equal(got.tokens, want.tokens) and np.array_equal(got.masked, want.masked), b
        assert np.array_equal(got.committed_now, want.committed_now) and got.fallback == want.fallback, b
        assert np.array_equal(got.conf, want.conf, equal_nan=True) and np.array_equal(got.argmax, want.argmax), b
    res = impl.unmask(lg, masked, tokens, 0.9, 2, 4, "bf16", seqs=[0, 2])
    assert res[1] is None and res[0] is not None and res[2] is not None
    # masked NLL: same marshalling
    tg = rng.integers(0, V, size=(B, S))
    nll, sums, counts = impl.masked_nll(lg, tg, masked, "bf16")
    for b in range(B):
        rows = np.full((S, V), np.nan)
        for p in range(S):
            if masked[b, p]:
                rows[p] = dec(lg[b, p])
        wn, wt, wc = impl.masked_nll_seq(rows, tg[b], masked[b].astype(bool))
        assert np.array_equal(nll[b], wn, equal_nan=True) and sums[b] == wt and counts[b] == wc, b
    nll2, sums2, counts2 = impl.masked_nll(lg, tg, masked, "bf16", seqs=[1])
    assert np.isnan(nll2[[0, 2]]).all() and np.isnan(sums2[[0, 2]]).all() and (counts2[[0, 2]] == -1).all()
    assert counts2[1] == 0 and sums2[1] == 0.0


ALL_CHECKS = [check_attention_bruteforce, check_attention_sdpa, check_attention_closed_forms,
              check_attention_invariants, check_attention_segment_merge, check_causal_block_bruteforce, check_causal_block_sdpa,
              check_causal_block_closed_forms, check_causal_block_invariants, check_unmask_closed_forms, check_unmask_bruteforce,
              check_unmask_rules, check_block_loop, check_append, check_linear_schedule,
              check_masked_nll_closed_forms, check_masked_nll_library, check_masked_nll_invariants,
              check_decode, check_commit_rule, check_batched_wrappers]
