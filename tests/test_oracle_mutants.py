"""Plant plausible mistakes in copies of the oracle and check that the pins catch each one.

The mistakes live only in this file, on the CPU; the oracle itself is untouched.
"""
import types

import numpy as np
import pytest

import oracle
from tests import oracle_pins


def _attention_mutant(kind):
    def attn(q, k_ctx, v_ctx, k_blk, v_blk, sm_scale, key_bias=None, return_probs=False, causal_block=False):
        S, Hq, D = q.shape
        Hkv = k_blk.shape[1]
        G = Hq // Hkv
        if kind == "drop_block":
            K, Vv = k_ctx, v_ctx
            if K.shape[0] == 0:
                K, Vv = k_blk[:1], v_blk[:1]
        elif kind == "drop_context":
            K, Vv = k_blk, v_blk
        else:
            K = np.concatenate([k_ctx, k_blk], axis=0)
            Vv = np.concatenate([v_ctx, v_blk], axis=0)
        if kind == "causal_block":
            pass
        o = np.empty((S, Hq, D))
        lse = np.empty((Hq, S))
        probs = np.empty((Hq, S, K.shape[0])) if return_probs else None
        for h in range(Hq):
            g = h % Hkv if kind == "gqa_modulo" else h // G
            sc = 1.0 if kind == "no_scale" else sm_scale
            s = sc * (q[:, h, :] @ K[:, g, :].T)
            if key_bias is not None and kind not in ("drop_block", "drop_context"):
                s = s + key_bias[None, :]
            L = k_ctx.shape[0]
            if kind == "causal_block" or (causal_block and kind == "none"):
                for i in range(S):
                    s[i, L + i + 1:] = -np.inf
            elif causal_block and kind == "causal_strict":      # a query misses its own key
                for i in range(S):
                    s[i, L + i:] = -np.inf
            elif causal_block and kind == "causal_loose":       # one key too many
                for i in range(S):
                    s[i, L + i + 2:] = -np.inf
            elif causal_block and kind == "causal_top_left":    # triangle over [context ; block]
                for i in range(S):
                    s[i, i + 1:] = -np.inf
            elif causal_block and kind == "causal_on_block_values_only":
                pass                                            # mask applied to P below instead
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            if kind == "wrong_axis":
                p = e / e.sum(axis=0, keepdims=True)
            else:
                p = e / e.sum(axis=1, keepdims=True)
            if causal_block and kind == "causal_on_block_values_only":
                # later block keys dropped after the normalisation (weights no longer sum to 1)
                for i in range(S):
                    p[i, L + i + 1:] = 0.0
            src = K if kind == "k_for_v" else Vv
            o[:, h, :] = p @ src[:, g, :]
            z = e.sum(axis=1)
            lse[h] = np.log(z) if kind == "lse_no_max" else m[:, 0] + np.log(z)
            if return_probs:
                probs[h] = p
        if return_probs:
            return o, lse, probs
        return o, lse
    return attn


def _context_rows_mutant(kind):
    def rows(pool, page_table_row, L, page_size):
        j = np.arange(L)
        if kind == "slot_off_by_one":
            pages = np.asarray(page_table_row)[j // page_size]
            slots = (j + 1) % page_size
        elif kind == "physical_order":
            pages = np.sort(np.asarray(page_table_row))[j // page_size] if L else np.zeros(0, int)
            slots = j % page_size
        else:
            pages = np.asarray(page_table_row)[j // page_size]
            slots = j % page_size
        return pool[pages, :, slots, :]
    return rows


def _unmask_mutant(kind):
    def unmask_seq(logits, masked, tokens, tau, step, T):
        S = masked.shape[0]
        masked = np.asarray(masked, dtype=bool)
        conf = np.full(S, np.nan)
        arg = np.full(S, -1, dtype=np.int64)
        for p in range(S):
            if not masked[p] and kind != "reread_locked":
                continue
            row = np.asarray(logits[p], dtype=np.float64)
            m = row.max()
            z = np.exp(row - m).sum()
            conf[p] = (np.exp(m) / z) if kind == "conf_wrong" else 1.0 / z
            if kind == "argmax_last":
                arg[p] = int(len(row) - 1 - np.argmax(row[::-1]))
            else:
                arg[p] = int(np.argmax(row))
        cand = [p for p in range(S) if masked[p]]
        chosen = [p for p in cand if conf[p] >= tau]
        fallback = False
        if step >= T and kind != "no_step_T":
            chosen = cand
        elif not chosen and cand and kind != "no_fallback":
            best = cand[0]
            for p in cand[1:]:
                if (conf[p] >= conf[best]) if kind == "fallback_last_tie" else (conf[p] > conf[best]):
                    best = p
            if kind == "fallback_least":
                best = min(cand, key=lambda p: conf[p])
            chosen = [best]
            fallback = True
        new_tokens = np.array(tokens, dtype=np.int64, copy=True)
        new_masked = masked.copy()
        committed = np.zeros(S, dtype=bool)
        for p in chosen:
            if kind != "no_token_write":
                new_tokens[p] = arg[p]
            new_masked[p] = False
            committed[p] = True
        if kind == "reread_locked":
            for p in range(S):
                if not masked[p] and np.isfinite(conf[p]) and conf[p] >= tau:
                    new_tokens[p] = arg[p]
        return oracle.UnmaskResult(new_tokens, new_masked, committed, conf, arg, fallback)
    return unmask_seq


def _append_mutant(kind):
    def kv_append(k_pool, v_pool, page_table, ctx_len, k_new, v_new, page_size, active=None):
        B, S = k_new.shape[:2]
        new_len = np.array(ctx_len, dtype=np.int64, copy=True)
        for b in range(B):
            if active is not None and not active[b] and kind != "ignore_active":
                continue
            L = int(ctx_len[b])
            if L + S > page_table.shape[1] * page_size and kind != "no_capacity_check":
                raise ValueError("block does not fit")
            for s in range(S):
                j = L + s + (1 if kind == "slot_shift" else 0)
                if j >= page_table.shape[1] * page_size:
                    continue
                page = page_table[b, j // page_size]
                k_pool[page, :, j % page_size, :] = k_new[b, s]
                v_pool[page, :, j % page_size, :] = (k_new if kind == "k_into_v" else v_new)[b, s]
            new_len[b] = L if kind == "no_len_update" else L + S
        return new_len
    return kv_append


def _schedule_mutant(kind):
    def mask(u, t):
        if not 0.0 <= t <= 1.0:
            if kind != "no_range_check":
                raise ValueError(t)
        u = np.asarray(u, dtype=np.float64)
        if kind == "inverted":            # keeps with probability t instead of masking
            return u >= t
        if kind == "one_minus_t":
            return u < 1.0 - t
        if kind == "quadratic":
            return u < t * t
        return u < t
    return mask


def _nll_mutant(kind):
    def nll_seq(logits, targets, masked):
        S = len(masked)
        nll = np.full(S, np.nan)
        total, count = 0.0, 0
        for p in range(S):
            if not masked[p] and kind != "include_unmasked":
                continue
            row = np.asarray(logits[p], dtype=np.float64)
            m = 0.0 if kind == "no_max_shift" else row.max()
            lse = m + np.log(np.exp(row - m).sum())
            tgt = int(targets[p]) + (1 if kind == "target_off_by_one" else 0)
            tgt = min(tgt, row.shape[0] - 1)
            if kind == "wrong_sign":
                nll[p] = row[tgt] - lse
            elif kind == "max_not_lse":
                nll[p] = m - row[tgt]
            else:
                nll[p] = lse - row[tgt]
            total += nll[p]
            count += 1
        if kind == "count_all":
            count = S
        return nll, total, count
    return nll_seq


def _decode_mutant(kind):
    def decode(x, dtype):
        if dtype == "bf16":
            if kind == "sign_extend":            # the 16-bit pattern taken as a signed integer
                bits = np.asarray(x).astype(np.uint16).view(np.int16).astype(np.int32) >> 0
                bits = (bits.astype(np.int64) << 16).astype(np.uint32) | \
                    (np.uint32(0xFFFF) * (bits < 0)).astype(np.uint32)   # ones smeared into the low half
                return bits.view(np.float32).astype(np.float64)
            shift = 15 if kind == "shift_15" else 16
            bits = np.asarray(x).astype(np.uint32) << np.uint32(shift)
            if kind == "low_half":               # the pattern read as the low half of a float32
                bits = np.asarray(x).astype(np.uint32)
            return bits.view(np.float32).astype(np.float64)
        if kind == "f32_via_bf16":               # float32 storage truncated to bf16 precision
            u = np.asarray(x, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
            return u.view(np.float32).astype(np.float64)
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    return decode


def _commit_rule_mutant(kind):
    def rule(conf, masked, tau, step, T):
        S = len(masked)
        masked = np.asarray(masked, dtype=bool)
        cand = [p for p in range(S) if masked[p]]
        if kind == "strict":
            chosen = [p for p in cand if conf[p] > tau]
        elif kind == "reads_locked":
            chosen = [p for p in range(S) if conf[p] >= tau]
        else:
            chosen = [p for p in cand if conf[p] >= tau]
        fallback = False
        if step >= T and kind != "no_step_T":
            chosen = cand
        elif not chosen and cand:
            best = cand[0]
            for p in cand[1:]:
                if (conf[p] >= conf[best]) if kind == "tie_last" else (conf[p] > conf[best]):
                    best = p
            chosen = [best]
            fallback = True
        committed = np.zeros(S, dtype=bool)
        committed[chosen] = True
        return committed, fallback
    return rule


def _batched_attention_mutant(kind):
    def denoise_attention(k_pool, v_pool, page_table, ctx_len, page_size, q, k_blk, v_blk, sm_scale, dtype,
                          seqs=None, causal_block=False):
        B, S, Hq, D = q.shape
        o = np.full((B, S, Hq, D), np.nan)
        lse = np.full((B, Hq, S), np.nan)
        for b in (range(B) if seqs is None or kind == "ignore_seqs" else seqs):
            L = int(ctx_len[b])
            tb = page_table[(b + 1) % B] if kind == "next_table" else page_table[b]
            if kind == "len_minus_one":
                L = max(0, L - 1)
            kc = oracle.decode(oracle.context_rows(k_pool, tb, L, page_size), dtype)
            vc = oracle.decode(oracle.context_rows((k_pool if kind == "k_pool_twice" else v_pool), tb, L,
                                                   page_size), dtype)
            o[b], lse[b] = oracle.denoise_attention_seq(oracle.decode(q[b], dtype), kc, vc,
                                                        oracle.decode(k_blk[b], dtype),
                                                        oracle.decode(v_blk[b], dtype), sm_scale,
                                                        causal_block=causal_block)
        return o, lse
    return denoise_attention


def _batched_unmask_mutant(kind):
    def unmask(logits, masked, tokens, tau, step, T, dtype, seqs=None):
        B = logits.shape[0]
        res = []
        for b in range(B):
            if seqs is not None and b not in seqs and kind != "ignore_seqs":
                res.append(None)
                continue
            lg = np.full((logits.shape[1], logits.shape[2]), np.nan)
            for p in range(logits.shape[1]):
                if masked[b, p]:
                    lg[p] = oracle.decode(logits[(b + 1) % B if kind == "next_row" else b, p], dtype)
            res.append(oracle.unmask_seq(lg, masked[b], tokens[0] if kind == "first_tokens" else tokens[b],
                                         tau, step, T))
        return res
    return unmask


def _batched_nll_mutant(kind):
    def masked_nll(logits, targets, masked, dtype, seqs=None):
        B, S = masked.shape
        nll = np.full((B, S), np.nan)
        sums = np.full(B, np.nan)
        counts = np.full(B, -1, dtype=np.int64)
        for b in (range(B) if seqs is None else seqs):
            lg = np.full((S, logits.shape[2]), np.nan)
            for p in range(S):
                if masked[b, p]:
                    lg[p] = oracle.decode(logits[b, p], dtype)
            tg = targets[b][::-1] if kind == "targets_reversed" else targets[b]
            nll[b], sums[b], counts[b] = oracle.masked_nll_seq(lg, tg, masked[b])
            if kind == "mean_not_sum" and counts[b] > 0:
                sums[b] /= counts[b]
        return nll, sums, counts
    return masked_nll


def _impl(**override):
    ns = types.SimpleNamespace(decode=oracle.decode, context_rows=oracle.context_rows,
                               denoise_attention_seq=oracle.denoise_attention_seq,
                               denoise_attention=oracle.denoise_attention,
                               unmask_seq=oracle.unmask_seq, commit_rule=oracle.commit_rule,
                               unmask=oracle.unmask, kv_append=oracle.kv_append,
                               linear_schedule_mask=oracle.linear_schedule_mask,
                               masked_nll_seq=oracle.masked_nll_seq, masked_nll=oracle.masked_nll)
    for k, v in override.items():
        setattr(ns, k, v)
    return ns


MUTANTS = (
    [("attn_" + k, dict(denoise_attention_seq=_attention_mutant(k)))
     for k in ("gqa_modulo", "drop_block", "drop_context", "no_scale", "wrong_axis", "k_for_v",
               "lse_no_max", "causal_block", "causal_ignored", "causal_strict", "causal_loose",
               "causal_top_left", "causal_on_block_values_only")]
    + [("rows_" + k, dict(context_rows=_context_rows_mutant(k)))
       for k in ("slot_off_by_one", "physical_order")]
    + [("unmask_" + k, dict(unmask_seq=_unmask_mutant(k)))
       for k in ("conf_wrong", "argmax_last", "no_step_T", "no_fallback", "fallback_last_tie",
                 "fallback_least", "no_token_write", "reread_locked")]
    + [("append_" + k, dict(kv_append=_append_mutant(k)))
       for k in ("ignore_active", "no_capacity_check", "slot_shift", "k_into_v", "no_len_update")]
    + [("schedule_" + k, dict(linear_schedule_mask=_schedule_mutant(k)))
       for k in ("inverted", "one_minus_t", "quadratic", "no_range_check")]
    + [("nll_" + k, dict(masked_nll_seq=_nll_mutant(k)))
       for k in ("include_unmasked", "no_max_shift", "target_off_by_one", "wrong_sign", "max_not_lse",
                 "count_all")]
    + [("decode_" + k, dict(decode=_decode_mutant(k)))
       for k in ("sign_extend", "shift_15", "low_half", "f32_via_bf16")]
    + [("rule_" + k, dict(commit_rule=_commit_rule_mutant(k)))
       for k in ("strict", "reads_locked", "tie_last", "no_step_T")]
    + [("batched_attn_" + k, dict(denoise_attention=_batched_attention_mutant(k)))
       for k in ("ignore_seqs", "next_table", "len_minus_one", "k_pool_twice")]
    + [("batched_unmask_" + k, dict(unmask=_batched_unmask_mutant(k)))
       for k in ("ignore_seqs", "first_tokens", "next_row")]
    + [("batched_nll_" + k, dict(masked_nll=_batched_nll_mutant(k)))
       for k in ("targets_reversed", "mean_not_sum")]
)


def test_unmutated_copy_passes():
    impl = _impl(denoise_attention_seq=_attention_mutant("none"),
                 context_rows=_context_rows_mutant("none"), unmask_seq=_unmask_mutant("none"),
                 kv_append=_append_mutant("none"), linear_schedule_mask=_schedule_mutant("none"),
                 masked_nll_seq=_nll_mutant("none"), decode=_decode_mutant("none"),
                 commit_rule=_commit_rule_mutant("none"), denoise_attention=_batched_attention_mutant("none"),
                 unmask=_batched_unmask_mutant("none"), masked_nll=_batched_nll_mutant("none"))
    for check in oracle_pins.ALL_CHECKS:
        check(impl)


@pytest.mark.filterwarnings("ignore::RuntimeWarning")   # overflow / NaN is how some mistakes show
@pytest.mark.parametrize("name,override", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, override):
    impl = _impl(**override)
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(impl)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            caught.append(check.__name__)
    assert caught, f"mutant {name} passed every pin"
