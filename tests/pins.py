"""Checks that pin the float64 attention oracle to facts other than its own code.

Every check takes ``attn(q, k, v, causal, scale, rows=None) -> (O, lse)`` on
float64 arrays, q [B, H, Nq, d] and k, v [B, H, Nk, d] (causal: 0 / False no
mask, 1 / True keys j <= i, 2 keys j <= i + Nk - Nq), so the same checks run against the real oracle
(tests/test_oracle_pins.py) and against deliberately broken copies of it
(tests/test_oracle_mutants.py), which must each fail at least one check.

Sources of truth (none of them is the oracle's formula retyped):

* closed forms the definition reduces to: uniform softmax when every logit is
  equal (Q = 0 or scale = 0), a single visible key in causal row 0, constant V;
* invariants of softmax attention: weights are a probability vector (seen
  through V = identity), joint permutation of keys and values, a per-row logit
  shift, an orthogonal change of basis shared by Q and K;
* a brute-force row-by-row evaluation in pure Python without max subtraction;
* for Nq != Nk: the same closed forms with the visible-key counts of each mask,
  and the end-aligned mask as the last rows of self-attention over a longer
  query sequence;
* hand-worked examples stored in tests/golden/two_key_softmax.json.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _rand(shape, seed, scale=1.0):
    return _rng(seed).standard_normal(shape) * scale


def check_zero_query_is_mean(attn):
    """Q = 0: every logit is 0, so O_i = mean of the visible V rows, lse_i = ln(#keys)."""
    B, H, N, d = 2, 3, 37, 8
    q = np.zeros((B, H, N, d))
    k, v = _rand((B, H, N, d), 1), _rand((B, H, N, d), 2)
    o, lse = attn(q, k, v, False, 0.7)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.full((B, H, N), math.log(N)), rtol=0, atol=1e-12)
    o, lse = attn(q, k, v, True, 0.7)
    prefix = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    np.testing.assert_allclose(o, prefix, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, N + 1)), lse.shape),
                               rtol=0, atol=1e-12)


def check_zero_scale_is_mean(attn):
    """scale = 0 with arbitrary Q, K: the same uniform average."""
    B, H, N, d = 1, 2, 19, 4
    q, k, v = (_rand((B, H, N, d), s, 3.0) for s in (3, 4, 5))
    o, lse = attn(q, k, v, False, 0.0)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape),
                               rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, math.log(N), rtol=0, atol=1e-12)


def check_causal_row0(attn):
    """Causal row 0 sees key 0 alone: O_0 = V_0 and lse_0 = its single logit."""
    B, H, N, d = 2, 2, 33, 16
    q, k, v = (_rand((B, H, N, d), s) for s in (6, 7, 8))
    scale = 0.3
    o, lse = attn(q, k, v, True, scale)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=0, atol=1e-12)
    single = scale * np.einsum("bhc,bhc->bh", q[:, :, 0], k[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], single, rtol=0, atol=1e-12)


def check_constant_v(attn):
    """V = c everywhere: every convex combination of V rows is c."""
    B, H, N, d = 1, 2, 45, 8
    q, k = _rand((B, H, N, d), 9, 2.0), _rand((B, H, N, d), 10, 2.0)
    c = _rand((d,), 11)
    v = np.broadcast_to(c, (B, H, N, d)).copy()
    for causal in (False, True):
        o, _ = attn(q, k, v, causal, 0.5)
        np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-12)


def check_weights_are_probabilities(attn):
    """V = identity (N = d) exposes the softmax weights as O: rows are probability
    vectors, and under the causal mask the weights above the diagonal are 0."""
    N = 24
    q, k = _rand((1, 2, N, N), 12), _rand((1, 2, N, N), 13)
    v = np.broadcast_to(np.eye(N), (1, 2, N, N)).copy()
    for causal in (False, True):
        o, _ = attn(q, k, v, causal, 0.4)
        assert np.all(o >= 0)
        np.testing.assert_allclose(o.sum(axis=-1), 1.0, rtol=0, atol=1e-12)
        if causal:
            upper = np.triu(np.ones((N, N), dtype=bool), 1)
            assert np.all(o[..., upper] == 0)
            assert np.all(o[..., ~upper] > 0)


def check_key_permutation(attn):
    """Non-causal attention is invariant to permuting keys and values together."""
    B, H, N, d = 1, 2, 50, 8
    q, k, v = (_rand((B, H, N, d), s) for s in (14, 15, 16))
    perm = _rng(17).permutation(N)
    o1, l1 = attn(q, k, v, False, 0.35)
    o2, l2 = attn(q, k[:, :, perm], v[:, :, perm], False, 0.35)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def check_logit_shift(attn):
    """Adding a constant a_i to every logit of row i leaves O unchanged and adds
    a_i to lse.  The shift is built by appending one feature: q' = [q, a/scale],
    k' = [k, 1] (and a zero column to V, dropped again)."""
    B, H, N, d = 1, 1, 29, 6
    q, k, v = (_rand((B, H, N, d), s) for s in (18, 19, 20))
    scale = 0.45
    a = _rand((B, H, N), 21, 5.0)
    q2 = np.concatenate([q, (a / scale)[..., None]], axis=-1)
    k2 = np.concatenate([k, np.ones((B, H, N, 1))], axis=-1)
    v2 = np.concatenate([v, np.zeros((B, H, N, 1))], axis=-1)
    for causal in (False, True):
        o1, l1 = attn(q, k, v, causal, scale)
        o2, l2 = attn(q2, k2, v2, causal, scale)
        np.testing.assert_allclose(o2[..., :d], o1, rtol=0, atol=1e-11)
        np.testing.assert_allclose(l2, l1 + a, rtol=0, atol=1e-11)


def check_orthogonal_invariance(attn):
    """Q M and K M with M orthogonal give the same logits, hence the same O, lse."""
    B, H, N, d = 1, 2, 40, 16
    q, k, v = (_rand((B, H, N, d), s) for s in (22, 23, 24))
    m, _ = np.linalg.qr(_rand((d, d), 25))
    for causal in (False, True):
        o1, l1 = attn(q, k, v, causal, 0.25)
        o2, l2 = attn(q @ m, k @ m, v, causal, 0.25)
        np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-11)
        np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-11)


def visible_keys(i, Nq, Nk, causal):
    """Number of keys query row i sees (keys 0 .. count-1)."""
    if int(causal) == 1:
        return min(i + 1, Nk)
    if int(causal) == 2:
        return i + 1 + (Nk - Nq)
    return Nk


def brute_force(q, k, v, causal, scale):
    """Row by row in pure Python: weights exp(s) with no max subtraction
    (inputs keep |s| small), normalised by their plain sum."""
    B, H, N, d = q.shape
    Nk = k.shape[2]
    o = np.zeros((B, H, N, d))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                keys = range(visible_keys(i, N, Nk, causal))
                weights = []
                for j in keys:
                    s = scale * sum(float(q[b, h, i, c]) * float(k[b, h, j, c]) for c in range(d))
                    weights.append(math.exp(s))
                total = sum(weights)
                for c in range(d):
                    o[b, h, i, c] = sum(w * float(v[b, h, j, c]) for w, j in zip(weights, keys)) / total
                lse[b, h, i] = math.log(total)
    return o, lse


def check_brute_force(attn):
    """Tiny non-square cases (N != d) against the pure-Python evaluation."""
    for (B, H, N, d), seed in (((1, 1, 1, 1), 30), ((1, 2, 7, 3), 31), ((2, 1, 16, 8), 32),
                               ((1, 1, 11, 5), 33)):
        q, k, v = (_rand((B, H, N, d), seed + 100 * s) for s in range(3))
        scale = 0.9 / math.sqrt(d)
        for causal in (False, True):
            o, lse = attn(q, k, v, causal, scale)
            ob, lb = brute_force(q, k, v, causal, scale)
            np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-12)


def check_brute_force_cross(attn):
    """Nq != Nk (and the end-aligned mask at Nq = Nk) against the pure-Python
    evaluation."""
    for (B, H, Nq, Nk, d), seed in (((1, 2, 5, 9, 3), 34), ((2, 1, 9, 5, 4), 35),
                                    ((1, 1, 1, 7, 2), 36), ((1, 1, 6, 6, 3), 37)):
        q = _rand((B, H, Nq, d), seed)
        k, v = _rand((B, H, Nk, d), seed + 100), _rand((B, H, Nk, d), seed + 200)
        scale = 0.8 / math.sqrt(d)
        for causal in (0, 1, 2):
            if causal == 2 and Nq > Nk:
                continue
            o, lse = attn(q, k, v, causal, scale)
            ob, lb = brute_force(q, k, v, causal, scale)
            np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-12)


def check_cross_zero_query(attn):
    """Q = 0 with Nq != Nk: O_i is the mean of the V rows row i sees and lse_i
    the log of their count, for each mask (counts counted here by hand: all Nk;
    min(i+1, Nk) from the start; i+1+Nk-Nq from the end)."""
    B, H, d = 2, 2, 4
    for Nq, Nk in ((13, 29), (29, 13), (1, 5)):
        q = np.zeros((B, H, Nq, d))
        k, v = _rand((B, H, Nk, d), 50 + Nq), _rand((B, H, Nk, d), 60 + Nq)
        for causal in (0, 1, 2):
            if causal == 2 and Nq > Nk:
                continue
            o, lse = attn(q, k, v, causal, 0.6)
            for i in range(Nq):
                n = {0: Nk, 1: min(i + 1, Nk), 2: i + 1 + Nk - Nq}[causal]
                np.testing.assert_allclose(o[:, :, i], v[:, :, :n].mean(axis=2), rtol=0, atol=1e-12)
                np.testing.assert_allclose(lse[:, :, i], math.log(n), rtol=0, atol=1e-12)


def check_end_aligned_is_suffix_of_self_attention(attn):
    """Causal mask aligned at the end: the Nq queries are the last Nq positions
    of an Nk-long sequence, so their rows equal the last Nq rows of causal
    self-attention of [X; Q] over the same keys, whatever X is."""
    B, H, Nq, Nk, d = 1, 2, 7, 20, 5
    q = _rand((B, H, Nq, d), 70)
    x = _rand((B, H, Nk - Nq, d), 71, 4.0)
    k, v = _rand((B, H, Nk, d), 72), _rand((B, H, Nk, d), 73)
    o, lse = attn(q, k, v, 2, 0.5)
    o_self, lse_self = attn(np.concatenate([x, q], axis=2), k, v, 1, 0.5)
    np.testing.assert_allclose(o, o_self[:, :, Nk - Nq:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_self[:, :, Nk - Nq:], rtol=0, atol=1e-12)


def check_rotary_complex(rot):
    """``rot(x, cos, sin, interleaved) -> out`` against RoFormer's definition: a
    feature pair read as the complex number a + ib is multiplied by e^{i phi}.
    Random angles per (position, pair); numpy's complex arithmetic on the same
    float32 table values."""
    B, H, N, d = 2, 3, 5, 8
    x = _rand((B, H, N, d), 80)
    phi = _rng(81).uniform(-np.pi, np.pi, (N, d // 2))
    c32, s32 = np.cos(phi).astype(np.float32), np.sin(phi).astype(np.float32)
    for interleaved in (False, True):
        out = rot(x, c32, s32, interleaved)
        ia = np.arange(0, d, 2) if interleaved else np.arange(d // 2)
        ib = ia + 1 if interleaved else ia + d // 2
        z = (x[..., ia] + 1j * x[..., ib]) * (c32.astype(np.float64) + 1j * s32.astype(np.float64))
        np.testing.assert_allclose(out[..., ia], z.real, rtol=0, atol=1e-14)
        np.testing.assert_allclose(out[..., ib], z.imag, rtol=0, atol=1e-14)


def check_golden(attn):
    """Hand-worked examples with exact expected values."""
    with open(os.path.join(GOLDEN, "two_key_softmax.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        q = np.array(case["q"], dtype=np.float64)[None, None]
        k = np.array(case["k"], dtype=np.float64)[None, None]
        v = np.array(case["v"], dtype=np.float64)[None, None]
        o, lse = attn(q, k, v, case["causal"], case["scale"])
        rows = case["rows_checked"]
        np.testing.assert_allclose(o[0, 0, rows], np.array(case["o"]), rtol=0, atol=1e-12,
                                   err_msg=case["name"])
        np.testing.assert_allclose(lse[0, 0, rows], np.array(case["lse"]), rtol=0, atol=1e-12,
                                   err_msg=case["name"])


def check_row_subset(attn):
    """Rows computed on their own equal the same rows of the full computation."""
    B, H, N, d = 1, 2, 31, 8
    q, k, v = (_rand((B, H, N, d), s) for s in (40, 41, 42))
    rows = np.array([0, 3, 17, 30])
    for causal in (False, True):
        o, lse = attn(q, k, v, causal, 0.3)
        os_, ls_ = attn(q, k, v, causal, 0.3, rows=rows)
        np.testing.assert_array_equal(os_, o[:, :, rows])
        np.testing.assert_array_equal(ls_, lse[:, :, rows])


ALL_CHECKS = [check_zero_query_is_mean, check_zero_scale_is_mean, check_causal_row0,
              check_constant_v, check_weights_are_probabilities, check_key_permutation,
              check_logit_shift, check_orthogonal_invariance, check_brute_force,
              check_golden, check_row_subset, check_brute_force_cross, check_cross_zero_query,
              check_end_aligned_is_suffix_of_self_attention]


# ------------------------------------------------------------------ backward
# Each check takes ``attn`` as above and ``bwd(q, k, v, g, causal, scale) ->
# (dQ, dK, dV)``, the gradients for dL/dO = g.

def _loss(attn, q, k, v, g, causal, scale):
    o, _ = attn(q, k, v, causal, scale)
    return float(np.sum(o * g))


def check_bwd_finite_differences(attn, bwd):
    """Every entry of dQ, dK, dV against central differences of L = sum(G * O)
    through the forward oracle (step 1e-5: truncation ~1e-10, rounding
    ~1e-11), for no mask and both causal alignments, Nq != Nk."""
    eps = 1e-5
    for (B, H, Nq, Nk, d), causal, seed in (((1, 2, 4, 6, 3), 0, 90), ((1, 1, 5, 5, 2), 1, 91),
                                            ((1, 1, 3, 6, 3), 2, 92), ((1, 1, 6, 4, 2), 1, 93)):
        q = _rand((B, H, Nq, d), seed)
        k, v = _rand((B, H, Nk, d), seed + 1), _rand((B, H, Nk, d), seed + 2)
        g = _rand((B, H, Nq, d), seed + 3)
        scale = 0.7
        grads = bwd(q, k, v, g, causal, scale)
        for which, (x, dx) in enumerate(zip((q, k, v), grads)):
            num = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                args = [q.copy(), k.copy(), v.copy()]
                args[which][idx] += eps
                up = _loss(attn, *args, g, causal, scale)
                args[which][idx] -= 2 * eps
                down = _loss(attn, *args, g, causal, scale)
                num[idx] = (up - down) / (2 * eps)
            np.testing.assert_allclose(dx, num, rtol=0, atol=1e-7)


def check_bwd_sums(attn, bwd):
    """Rows of the softmax Jacobian sum to zero, so the key gradients of a head
    sum to zero; rows of P sum to one, so the value gradients sum to the
    summed output gradient."""
    B, H, Nq, Nk, d = 2, 2, 9, 13, 4
    q = _rand((B, H, Nq, d), 94)
    k, v = _rand((B, H, Nk, d), 95), _rand((B, H, Nk, d), 96)
    g = _rand((B, H, Nq, d), 97)
    for causal in (0, 1, 2):
        _, dk, dv = bwd(q, k, v, g, causal, 0.5)
        np.testing.assert_allclose(dk.sum(axis=2), 0.0, rtol=0, atol=1e-12)
        np.testing.assert_allclose(dv.sum(axis=2), g.sum(axis=2), rtol=0, atol=1e-12)


def check_bwd_zero_scale(attn, bwd):
    """scale = 0: every logit is 0, so dQ = dK = 0 and dV_j is the sum over
    the rows that see key j of g_i / (number of keys row i sees)."""
    B, H, Nq, Nk, d = 1, 2, 6, 8, 3
    q = _rand((B, H, Nq, d), 98)
    k, v = _rand((B, H, Nk, d), 99), _rand((B, H, Nk, d), 100)
    g = _rand((B, H, Nq, d), 101)
    for causal in (0, 1, 2):
        dq, dk, dv = bwd(q, k, v, g, causal, 0.0)
        assert np.all(dq == 0) and np.all(dk == 0)
        want = np.zeros_like(v)
        for i in range(Nq):
            n = visible_keys(i, Nq, Nk, causal)
            want[:, :, :n] += g[:, :, i:i + 1] / n
        np.testing.assert_allclose(dv, want, rtol=0, atol=1e-13)


def check_bwd_unseen_keys_get_nothing(attn, bwd):
    """Top-left causal mask with Nq < Nk: keys j >= Nq are seen by no row, so
    their gradients are exactly zero; the zero output gradient gives zero
    gradients everywhere."""
    B, H, Nq, Nk, d = 1, 1, 4, 9, 3
    q = _rand((B, H, Nq, d), 102)
    k, v = _rand((B, H, Nk, d), 103), _rand((B, H, Nk, d), 104)
    g = _rand((B, H, Nq, d), 105)
    _, dk, dv = bwd(q, k, v, g, 1, 0.8)
    assert np.all(dk[:, :, Nq:] == 0) and np.all(dv[:, :, Nq:] == 0)
    assert np.any(dk[:, :, :Nq] != 0) and np.any(dv[:, :, :Nq] != 0)
    for x in bwd(q, k, v, np.zeros_like(g), 0, 0.8):
        assert np.all(x == 0)


def check_bwd_golden(attn, bwd):
    """Hand-worked gradients with exact expected values
    (tests/golden/two_key_backward.json)."""
    with open(os.path.join(GOLDEN, "two_key_backward.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        q, k, v, g = (np.array(case[n], dtype=np.float64)[None, None] for n in ("q", "k", "v", "g"))
        grads = bwd(q, k, v, g, 1 if case["causal"] else 0, case["scale"])
        for name, got in zip(("dq", "dk", "dv"), grads):
            np.testing.assert_allclose(got[0, 0], np.array(case[name]), rtol=0, atol=1e-14,
                                       err_msg=f"{case['name']}: {name}")


BWD_CHECKS = [check_bwd_finite_differences, check_bwd_sums, check_bwd_zero_scale,
              check_bwd_unseen_keys_get_nothing, check_bwd_golden]
