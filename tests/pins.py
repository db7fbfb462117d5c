"""Pins of the float64 oracle against facts it does not compute itself.

Each ``pin_*`` function takes a loaded ``oracle.Oracle`` and raises
``AssertionError`` on a mismatch.  ``test_oracle_pins.py`` runs them against
the real oracle; ``test_oracle_mutants.py`` runs them against copies of the
oracle with one planted mistake each and requires that some pin fails.

The facts used:
  * IEEE-754 rounding to nearest-even, checked by comparing the two
    neighbouring representable values (bf16) and numpy's float16 cast (fp16);
  * the quantiser's error bound |x - s*code| <= s/2 and code round trip;
  * closed forms: one visible position returns its V, equal scores return the
    mean of V, a zero query returns the mean, hand-derived golden cases;
  * invariances: a constant added to every key, permuting positions;
  * softmax weights summing to one; the large-score limit;
  * GQA: kv head h // group, and equality with MHA on repeated K/V;
  * a pure-Python brute force (``oracle/brute.py``) on tiny decode steps;
  * a step of T new tokens equals T single-token steps in a row;
  * the output projection: the brute force on a non-square weight, a weight
    whose rows are unit vectors (y picks entries of x), linearity in x.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

from oracle import brute
from synthetic import WORKLOADS, Workload, gen_all, to_storage

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_forms.json")


# ---------------------------------------------------------------- storage
def pin_bf16_rounding(o):
    rng = np.random.default_rng(100)
    vals = np.concatenate([
        rng.standard_normal(400).astype(np.float32),
        (rng.standard_normal(200) * 1e-3).astype(np.float32),
        (rng.standard_normal(200) * 1e30).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40, -1e-41], np.float32),
    ])
    # exact ties: low 16 bits = 0x8000, with even and odd kept halves
    ties = (rng.integers(0x0080, 0x7F00, 64, dtype=np.uint32) << 16) | 0x8000
    vals = np.concatenate([vals, ties.view(np.float32), (ties | 0x80000000).view(np.float32)])
    got = o.f32_to_bf16(vals)
    want = np.array([brute._bf16_nearest(v) for v in vals], np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"bf16 rounding differs at {vals[bad[:4]]}: {got[bad[:4]]} vs {want[bad[:4]]}"
    bits = rng.integers(0, 0x7F80, 256).astype(np.uint16)
    dec = o.bf16_to_f32(bits)
    assert np.array_equal(dec.view(np.uint32), bits.astype(np.uint32) << 16), "bf16 decode"


def pin_f16_rounding(o):
    rng = np.random.default_rng(101)
    vals = np.concatenate([
        rng.standard_normal(400).astype(np.float32),
        (rng.standard_normal(200) * 1e-5).astype(np.float32),   # fp16 subnormals
        (rng.standard_normal(100) * 3e4).astype(np.float32),    # near the fp16 maximum
        np.array([0.0, -0.0, 65504.0, 65520.0, 1e-8, 2.0 ** -25], np.float32),
    ])
    got = o.f32_to_f16(vals)
    with np.errstate(over="ignore"):
        want = vals.astype(np.float16).view(np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"fp16 rounding differs at {vals[bad[:4]]}"
    bits = rng.integers(0, 0x7C00, 256).astype(np.uint16)
    assert np.array_equal(o.f16_to_f32(bits), bits.view(np.float16).astype(np.float32)), "fp16 decode"


def pin_quant_i8(o):
    rng = np.random.default_rng(102)
    for trial in range(200):
        D = int(rng.choice([1, 7, 64, 128]))
        x = (rng.standard_normal(D) * rng.uniform(1e-3, 10)).astype(np.float32)
        code, s = o.quant_i8(x)
        amax = float(np.max(np.abs(x)))
        assert s > 0 and abs(s - amax / 127.0) <= 1e-6 * s, f"scale {s} vs absmax/127 {amax / 127}"
        assert code.min() >= -127 and code.max() <= 127
        err = np.abs(x.astype(np.float64) - s * code.astype(np.float64))
        assert np.all(err <= s * (0.5 + 1e-5)), f"|x - s*code| > s/2: {err.max()} vs {s / 2}"
        i = int(np.argmax(np.abs(x)))
        assert abs(int(code[i])) == 127, "absmax element must map to +-127"
        assert np.sign(code[i]) == np.sign(x[i])
        # dequantise and quantise again: the codes come back unchanged
        code2, _ = o.quant_i8((np.float32(s) * code.astype(np.float32)).astype(np.float32))
        assert np.array_equal(code, code2), "int8 round trip"
    code, s = o.quant_i8(np.zeros(16, np.float32))
    assert s == 1.0 and not code.any(), "all-zero row -> scale 1, codes 0"


# --------------------------------------------------------------- attention
def pin_attend_closed_forms(o):
    rng = np.random.default_rng(103)
    D = 16
    V = rng.standard_normal((5, D))
    # one visible row returns it exactly
    out, p = o.attend(rng.standard_normal(D), rng.standard_normal((1, D)), V[:1], 0.25)
    assert np.array_equal(out, V[0]) and p[0] == 1.0, "single position must return V0"
    # identical keys -> uniform weights -> mean of V
    K = np.tile(rng.standard_normal(D), (5, 1))
    out, p = o.attend(rng.standard_normal(D), K, V, 0.25)
    assert np.allclose(out, V.mean(0), rtol=0, atol=1e-13), "identical keys -> mean(V)"
    # zero query -> mean of V
    out, _ = o.attend(np.zeros(D), rng.standard_normal((5, D)), V, 0.25)
    assert np.allclose(out, V.mean(0), rtol=0, atol=1e-13), "q = 0 -> mean(V)"
    # two positions, scores differing by ln 3 -> (3/4, 1/4)
    q = np.zeros(D); q[0] = math.log(3.0) / 0.5
    K2 = np.zeros((2, D)); K2[0, 0] = 1.0
    out, p = o.attend(q, K2, V[:2], 0.5)
    assert abs(p[0] - 0.75) < 1e-14 and abs(p[1] - 0.25) < 1e-14, f"p = {p}"
    assert np.allclose(out, 0.75 * V[0] + 0.25 * V[1], atol=1e-14)
    # order of q.K: scores must use q against each key, scaled once
    q = rng.standard_normal(D); K = rng.standard_normal((7, D)); V7 = rng.standard_normal((7, D))
    s = 0.3 * (K @ q)
    w = np.exp(s - s.max())
    pw = w / w.sum()
    out, p = o.attend(q, K, V7, 0.3)
    assert np.allclose(p, pw, rtol=1e-12, atol=0) and np.allclose(out, pw @ V7, rtol=1e-11, atol=1e-14)


def pin_attend_invariants(o):
    rng = np.random.default_rng(104)
    for n, D in [(1, 8), (3, 16), (50, 64), (300, 128)]:
        q = rng.standard_normal(D); K = rng.standard_normal((n, D)); V = rng.standard_normal((n, D))
        out, p = o.attend(q, K, V, 1 / math.sqrt(D))
        assert abs(p.sum() - 1.0) <= 1e-12, "softmax weights must sum to 1"
        assert np.all(p >= 0)
        c = rng.standard_normal(D) * 3
        out2, _ = o.attend(q, K + c, V, 1 / math.sqrt(D))
        assert np.allclose(out, out2, rtol=1e-10, atol=1e-12), "shift of all keys must not change o"
        perm = rng.permutation(n)
        out3, _ = o.attend(q, K[perm], V[perm], 1 / math.sqrt(D))
        assert np.allclose(out, out3, rtol=1e-10, atol=1e-12), "permuting positions must not change o"
        # large-score limit: o -> V at the argmax, stays finite
        out4, p4 = o.attend(q * 1e3, K, V, 1 / math.sqrt(D))
        t = int(np.argmax(K @ q))
        assert np.all(np.isfinite(out4)) and np.allclose(out4, V[t], atol=1e-6), "large-score limit"


# ----------------------------------------------------------- full decode step
def _bf(bits):
    """bfloat16 bit patterns -> float32 values (the upper half of binary32)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _small(cache="f32", qkv="f32", B=2, Hq=4, Hkv=2, D=8, Lmax=16, lens=(5, 11), bias=0.1, seed=7, q_len=1):
    w = Workload("pin", B=B, Hq=Hq, Hkv=Hkv, D=D, Lmax=Lmax, qkv_dtype=qkv, cache_dtype=cache,
                 lens=("fixed", 0), bias_std=bias, seed=seed, q_len=q_len)
    inp = gen_all(w, seed=seed, seq_lens=np.array(lens, np.int32), fill_beyond="nan")
    return w, inp


def pin_brute_force(o):
    cases = [
        dict(cache="f32", qkv="f32"),
        dict(cache="f16", qkv="f16"),
        dict(cache="bf16", qkv="bf16"),
        dict(cache="bf16", qkv="f32", bias=None),
        dict(cache="i8", qkv="f16"),
        dict(cache="f16", qkv="bf16", Hq=4, Hkv=1, lens=(0, 15)),
        dict(cache="bf16", qkv="bf16", B=3, Hq=2, Hkv=2, lens=(-1, 3, 16)),
    ]
    for kw in cases:
        w, inp = _small(**kw)
        a = o.decode_step(w, inp)
        b = brute.decode_step(w, inp)
        assert a["overflow"] == b["overflow"], f"overflow flag {kw}"
        assert np.array_equal(a["k_cache"].view(np.uint8), b["k_cache"].view(np.uint8)), f"k append {kw}"
        assert np.array_equal(a["v_cache"].view(np.uint8), b["v_cache"].view(np.uint8)), f"v append {kw}"
        if w.cache_dtype == "i8":
            assert np.array_equal(a["scales"].view(np.uint32), b["scales"].view(np.uint32)), "scales"
        err = np.max(np.abs(a["out"] - b["out"]))
        assert err <= 1e-12, f"oracle vs brute force {kw}: {err}"


def pin_append_semantics(o):
    w, inp = _small(cache="bf16", qkv="bf16", B=4, lens=(0, 7, -1, 16))
    r = o.decode_step(w, inp)
    assert r["overflow"], "seq_lens >= Lmax must raise the overflow flag"
    kc0, kc1 = inp["k_cache"], r["k_cache"]
    for b, L in enumerate(inp["seq_lens"]):
        changed = np.nonzero(np.any(kc0[b] != kc1[b], axis=(0, 2)))[0]
        if 0 <= L < w.Lmax:
            assert list(changed) == [L], f"slot {b}: append touched rows {changed}, expected [{L}]"
            k32 = _bf(inp["k_new"][b]) + _bf(inp["bias"][w.Hq * w.D:(w.Hq + w.Hkv) * w.D]).reshape(w.Hkv, w.D)
            want = to_storage(k32, "bf16")
            assert np.array_equal(kc1[b, :, L, :], want), f"slot {b}: appended row"
        else:
            assert changed.size == 0, f"slot {b} (L={L}) must leave the cache untouched"
            assert not r["out"][b].any(), f"slot {b} (L={L}) must give zeros"
    # the single visible position of slot 0 is the new token itself
    kvh = np.arange(w.Hq) // w.group
    v_row = _bf(r["v_cache"][0, :, 0, :]).astype(np.float64)
    assert np.array_equal(r["out"][0], v_row[kvh]), "ctx 1 -> V"


def pin_gqa_mapping(o):
    w, inp = _small(cache="f32", qkv="f32", B=2, Hq=6, Hkv=2, D=8, lens=(9, 4), bias=None)
    r = o.decode_step(w, inp)
    # MHA on K/V repeated per group must agree
    wm = w.with_(Hkv=6)
    inp_m = dict(inp)
    rep = lambda a: np.repeat(a, 3, axis=1)
    inp_m.update(k_new=rep(inp["k_new"]), v_new=rep(inp["v_new"]), k_cache=rep(inp["k_cache"]),
                 v_cache=rep(inp["v_cache"]))
    rm = o.decode_step(wm, inp_m)
    assert np.allclose(r["out"], rm["out"], rtol=0, atol=1e-13), "GQA != MHA on repeated K/V"


def pin_golden(o):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        w = Workload(c["name"], B=c["B"], Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"], Lmax=c["Lmax"],
                     qkv_dtype="f32", cache_dtype="f32")
        L = c["seq_len"]
        kc = np.full((1, w.Hkv, w.Lmax, w.D), np.nan, np.float32)
        vc = np.full((1, w.Hkv, w.Lmax, w.D), np.nan, np.float32)
        kc[0, :, :L, :] = np.array(c["k_hist"], np.float32).reshape(w.Hkv, L, w.D)
        vc[0, :, :L, :] = np.array(c["v_hist"], np.float32).reshape(w.Hkv, L, w.D)
        inp = dict(q=np.array(c["q"], np.float32).reshape(1, w.Hq, w.D),
                   k_new=np.array(c["k_new"], np.float32).reshape(1, w.Hkv, w.D),
                   v_new=np.array(c["v_new"], np.float32).reshape(1, w.Hkv, w.D),
                   bias=None, k_cache=kc, v_cache=vc, seq_lens=np.array([L], np.int32))
        r = o.decode_step(w, inp, softmax_scale=c.get("scale", 0.0))
        got = r["out"].ravel()
        assert np.allclose(got, c["expect"], rtol=0, atol=c["tol"]), f"{c['name']}: {got} vs {c['expect']}"


def pin_workload_tiny(o):
    """The tiny workload end to end against the brute force."""
    w = WORKLOADS["tiny"]
    inp = gen_all(w)
    a = o.decode_step(w, inp)
    b = brute.decode_step(w, inp)
    assert np.max(np.abs(a["out"] - b["out"])) <= 1e-12
    assert np.array_equal(a["k_cache"], b["k_cache"]) and np.array_equal(a["v_cache"], b["v_cache"])


def pin_sliding_window(o):
    """A window covering the context changes nothing; a window of 1 returns the new V; brute force."""
    w, inp = _small(cache="bf16", qkv="bf16", B=3, Hq=4, Hkv=2, D=8, Lmax=32, lens=(20, 3, 31))
    full = o.decode_step(w, inp)
    assert np.array_equal(o.decode_step(w, inp, window=32)["out"], full["out"]), "window >= context"
    assert not np.array_equal(o.decode_step(w, inp, window=4)["out"], full["out"]), "window must matter"
    one = o.decode_step(w, inp, window=1)
    kvh = np.arange(w.Hq) // w.group
    for b, L in enumerate(inp["seq_lens"]):
        v_new = _bf(one["v_cache"][b, :, L, :]).astype(np.float64)
        assert np.array_equal(one["out"][b], v_new[kvh]), "window 1 -> the new token's V"
    for win in (2, 5, 17):
        a = o.decode_step(w, inp, window=win)
        bb = brute.decode_step(w, inp, window=win)
        assert np.max(np.abs(a["out"] - bb["out"])) <= 1e-12, f"window {win} vs brute force"


def _same_bytes(a, b):
    return np.array_equal(np.ascontiguousarray(a).view(np.uint8), np.ascontiguousarray(b).view(np.uint8))


def pin_multi_token(o):
    """T new tokens per step: brute force on tiny steps; equal to T single-token steps in a row;
    the overflow edge L + T = Lmax (fits) vs Lmax + 1 (flagged); a window of 1 returns each
    token's own V."""
    cases = [dict(cache="f32", qkv="f32", q_len=2, lens=(5, 13)),
             dict(cache="bf16", qkv="bf16", q_len=3, lens=(0, 12)),
             dict(cache="i8", qkv="f16", q_len=4, lens=(7, 1)),
             dict(cache="f16", qkv="f16", q_len=5, Hq=4, Hkv=1, lens=(10, 3))]
    for kw in cases:
        w, inp = _small(**kw)
        T = w.q_len
        a = o.decode_step(w, inp)
        bb = brute.decode_step(w, inp)
        assert a["out"].shape == (w.B, T, w.Hq, w.D)
        assert not a["overflow"] and not bb["overflow"], kw
        assert np.max(np.abs(a["out"] - bb["out"])) <= 1e-12, f"q_len vs brute force {kw}"
        assert _same_bytes(a["k_cache"], bb["k_cache"]) and _same_bytes(a["v_cache"], bb["v_cache"]), kw
        for win in (1, 3):
            aw = o.decode_step(w, inp, window=win)
            bw = brute.decode_step(w, inp, window=win)
            assert np.max(np.abs(aw["out"] - bw["out"])) <= 1e-12, f"q_len window {win} {kw}"
        # T single-token steps, each appending one token and advancing the lengths
        w1 = w.with_(q_len=1)
        cur = dict(inp)
        for j in range(T):
            step = dict(cur, q=inp["q"][:, j], k_new=inp["k_new"][:, j], v_new=inp["v_new"][:, j],
                        seq_lens=inp["seq_lens"] + j)
            r1 = o.decode_step(w1, step)
            assert np.max(np.abs(r1["out"] - a["out"][:, j])) <= 1e-13, f"token {j} vs single steps {kw}"
            cur = dict(cur, k_cache=r1["k_cache"], v_cache=r1["v_cache"], scales=r1["scales"])
        assert _same_bytes(cur["k_cache"], a["k_cache"]) and _same_bytes(cur["v_cache"], a["v_cache"]), kw
        if w.cache_dtype == "i8":
            assert _same_bytes(cur["scales"], a["scales"]), kw
    # the overflow edge: L + T = Lmax fits, Lmax + 1 does not
    w, inp = _small(cache="bf16", qkv="bf16", q_len=3, lens=(13, 14))
    r = o.decode_step(w, inp)
    assert r["overflow"], "L + T > Lmax must raise the overflow flag"
    assert r["out"][0].any() and not r["out"][1].any(), "slot 0 fits (13 + 3 = 16), slot 1 does not"
    assert _same_bytes(r["k_cache"][1], inp["k_cache"][1]), "an overflowing slot keeps its cache"
    # window 1: every token sees only itself
    w, inp = _small(cache="f32", qkv="f32", q_len=3, lens=(4, 9))
    one = o.decode_step(w, inp, window=1)
    kvh = np.arange(w.Hq) // w.group
    for b, L in enumerate(inp["seq_lens"]):
        for j in range(3):
            v = one["v_cache"][b, :, L + j, :].astype(np.float64)
            assert np.array_equal(one["out"][b, j], v[kvh]), "window 1 -> the token's own V"


def pin_out_proj(o):
    """The output projection y = x . W^T: equal to the pure-Python loops on a non-square W with
    distinct entries (a transposed or shifted index fails); W with unit-vector rows picks the
    entries of x; a zero W row gives zero; linear in x."""
    rng = np.random.default_rng(31)
    for n_tok, K, F in ((1, 5, 3), (3, 8, 11), (4, 16, 6)):
        x = rng.standard_normal((n_tok, K))
        W = rng.standard_normal((F, K))
        y = o.out_proj(x, W)
        assert y.shape == (n_tok, F)
        assert np.max(np.abs(y - np.array(brute.out_proj(x, W)))) <= 1e-12, (n_tok, K, F)
        x2 = rng.standard_normal((n_tok, K))
        assert np.max(np.abs(o.out_proj(x + 2.0 * x2, W) - (y + 2.0 * o.out_proj(x2, W)))) <= 1e-12
    # unit-vector rows: feature f reads element sel[f] of each token's row
    K, F = 12, 7
    sel = np.array([11, 0, 5, 5, 3, 10, 1])
    W = np.zeros((F, K))
    W[np.arange(F), sel] = 1.0
    W[2] = 0.0  # and a zero row
    x = rng.standard_normal((2, 3, 4))  # [B][Hq][D] flattened to K = 12 per token
    y = o.out_proj(x, W)
    flat = x.reshape(2, K)
    want = flat[:, sel].copy()
    want[:, 2] = 0.0
    assert np.array_equal(y, want), "unit-vector rows select entries of the flattened output"


ALL_PINS = [pin_bf16_rounding, pin_f16_rounding, pin_quant_i8, pin_attend_closed_forms,
            pin_attend_invariants, pin_brute_force, pin_append_semantics, pin_gqa_mapping,
            pin_golden, pin_workload_tiny, pin_sliding_window, pin_multi_token, pin_out_proj]
