"""Hand-worked examples (tests/golden/*.txt) against the float64 oracle."""
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
_ENV = {k: getattr(math, k) for k in ("exp", "log", "e", "sqrt")}


def _read(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            out[key.strip()] = [part.strip() for part in val.split(";")]
    return out


def _nums(parts):
    return np.array([[eval(x, {"__builtins__": {}}, _ENV) for x in p.split()] for p in parts], float)


def test_attention_worked_example():
    g = _read("attention_worked.txt")
    q = _nums(g["q"]).reshape(1, 1, 2)
    kc, vc = _nums(g["k_ctx"])[:, None, :], _nums(g["v_ctx"])[:, None, :]
    kb, vb = _nums(g["k_blk"])[:, None, :], _nums(g["v_blk"])[:, None, :]
    o, lse = oracle.denoise_attention_seq(q, kc, vc, kb, vb, 1.0)
    want_o = [eval(x, {"__builtins__": {}}, _ENV) for x in g["o"]]
    assert np.allclose(o[0, 0], want_o, rtol=1e-15, atol=0)
    assert abs(lse[0, 0] - eval(g["lse"][0], {"__builtins__": {}}, _ENV)) < 1e-15


def test_unmask_worked_example():
    g = _read("unmask_worked.txt")
    lg = _nums(g["logits"])
    want_conf = [eval(x, {"__builtins__": {}}, _ENV) for x in g["conf"]]
    masked = np.ones(3, bool)
    tokens = np.full(3, -1)
    for step in (1, 2, 3):
        r = oracle.unmask_seq(lg, masked, tokens, 0.9, step, 3)
        for p in range(3):
            if masked[p]:
                assert abs(r.conf[p] - want_conf[p]) < 1e-15
                assert r.argmax[p] == int(g["argmax"][0].split()[p])
        assert list(r.committed_now.astype(int)) == [int(x) for x in g[f"step{step}_committed"][0].split()]
        masked, tokens = r.masked, r.tokens
    assert list(tokens) == [int(x) for x in g["final_tokens"][0].split()]


def test_context_block_attention_worked_example():
    g = _read("context_block_attention_worked.txt")
    q = _nums(g["q"])[:, None, :]
    kc, vc = _nums(g["k_ctx"])[:, None, :], _nums(g["v_ctx"])[:, None, :]
    kb, vb = _nums(g["k_blk"])[:, None, :], _nums(g["v_blk"])[:, None, :]
    o, lse = oracle.denoise_attention_seq(q, kc, vc, kb, vb, 1.0, causal_block=True)
    for i in range(2):
        want_o = [eval(x, {"__builtins__": {}}, _ENV) for x in g[f"o{i}"]]
        assert np.allclose(o[i, 0], want_o, rtol=1e-15, atol=0), i
        assert abs(lse[0, i] - eval(g["lse"][i], {"__builtins__": {}}, _ENV)) < 1e-15, i
    # the denoise view differs at block position 0 (it also sees k2)
    ob, _ = oracle.denoise_attention_seq(q, kc, vc, kb, vb, 1.0)
    assert not np.allclose(ob[0, 0], o[0, 0])


def test_masked_nll_worked_example():
    g = _read("masked_nll_worked.txt")
    u = _nums(g["u"])[0]
    masked = oracle.linear_schedule_mask(u, float(g["t"][0]))
    assert list(masked.astype(int)) == [int(x) for x in g["masked"][0].split()]
    lg = _nums(g["logits"])
    tg = np.array([int(x) for x in g["targets"][0].split()])
    nll, tot, cnt = oracle.masked_nll_seq(lg, tg, masked)
    want = [eval(x, {"__builtins__": {}}, _ENV) for x in g["nll"]]
    assert cnt == 2 and np.isnan(nll[1])
    assert np.allclose(nll[[0, 2]], want, rtol=0, atol=1e-14)
    assert abs(tot - sum(want)) < 1e-14
