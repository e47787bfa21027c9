"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with something other than itself: a worked example printed on
a page, a closed form, an invariant of the definition, brute force on tiny
rows, finite differences, or an independent library routine.  The test module
runs them on the real oracle; the mutant test compiles the oracle with planted
mistakes and checks that every mistake fails at least one pin.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

from oracle import dropout_params as oracle_dropout_params

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition("=")
            parts = val.split()
            vals[key.strip()] = [float(p) for p in parts] if len(parts) > 1 else float(parts[0])
    return vals


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.abs(a - b)
    bound = atol + rtol * np.abs(b)
    if not np.all(err <= bound):
        i = int(np.argmax(err - bound))
        raise AssertionError(f"{what}: max excess at {i}: {a.reshape(-1)[i]!r} vs "
                             f"{b.reshape(-1)[i]!r} (err {err.reshape(-1)[i]:.3e})")


# ---------------------------------------------------------------- pin 1
def pin_worked_example(orc):
    """The page's worked online-softmax example (scores 1 2 3 0, blocks of two),
    "What is Flash Attention?" transcript 05:49-06:52, within the page's
    rounding; and the same numbers to 1e-12 against their closed forms."""
    g = _read_golden("online_softmax_worked_example.txt")
    x = np.array(g["scores"])
    m, l = orc.online_softmax(x, int(g["block"]))
    tol = g["page_tolerance"]
    assert m[0] == g["m1"] and m[1] == g["m2"], (m, g)
    _close(l[0], g["l1"], tol, what="l1 vs page")
    _close(l[1], g["l2"], tol, what="l2 vs page")
    alpha = math.exp(m[0] - m[1])
    _close(alpha, g["alpha"], tol, what="alpha vs page")
    _close(alpha * l[0], g["alpha_l1"], tol, what="alpha*l1 vs page")
    _close(l[1] - alpha * l[0], g["block2_sum"], tol, what="block-2 sum vs page")
    _close(l[1] / math.exp(-m[1]), g["denominator"], tol, what="denominator vs page")
    # closed forms
    _close(l[0], math.exp(-1.0) + 1.0, 1e-12, what="l1 closed form")
    denom = math.exp(1) + math.exp(2) + math.exp(3) + math.exp(0)
    _close(l[1], math.exp(-3.0) * denom, 1e-12, what="l2 closed form")
    # the same row through the definition: q = e_0, k_j = (s_j, 0, ...), v = I.
    q = np.zeros((1, 1, 4))
    q[0, 0, 0] = 1.0
    k = np.zeros((1, 4, 4))
    k[0, :, 0] = x
    v = np.eye(4).reshape(1, 4, 4)
    qq = np.repeat(q, 4, axis=1)  # every query row equal
    o, lse = orc.forward(qq, k, v, 1.0, False)
    p_exact = np.exp(x) / denom
    _close(o[0], p_exact, 1e-12, atol=1e-15, what="softmax of the worked row")
    _close(lse[0], math.log(denom), 1e-12, what="lse of the worked row")
    _close(lse[0], m[1] + math.log(l[1]), 1e-12, what="lse == m + ln l")


# ---------------------------------------------------------------- pin 2
def pin_zero_query(orc):
    """Q = 0 makes every visible score 0: O is the mean of the visible V rows
    and lse = ln(#visible)."""
    rng = _rng(2)
    BH, N, d = 3, 37, 8
    q = np.zeros((BH, N, d))
    k = rng.standard_normal((BH, N, d))
    v = rng.standard_normal((BH, N, d))
    o, lse = orc.forward(q, k, v, 0.3, False)
    _close(o.reshape(BH, N, d), np.broadcast_to(v.mean(axis=1, keepdims=True), (BH, N, d)),
           1e-12, atol=1e-14, what="Q=0 non-causal O")
    _close(lse, np.full(BH * N, math.log(N)), 1e-13, what="Q=0 non-causal lse")
    o, lse = orc.forward(q, k, v, 0.3, True)
    prefix = np.cumsum(v, axis=1) / np.arange(1, N + 1)[None, :, None]
    _close(o.reshape(BH, N, d), prefix, 1e-12, atol=1e-14, what="Q=0 causal O")
    _close(lse.reshape(BH, N), np.broadcast_to(np.log(np.arange(1, N + 1)), (BH, N)), 1e-13,
           atol=1e-15, what="Q=0 causal lse")


# ---------------------------------------------------------------- pin 3
def pin_one_hot(orc):
    """q_i = c e_1, k_{j*} = e_1, other keys orthogonal to e_1, c*scale = 40:
    O_i = v_{j*} up to N e^{-40} max|v|."""
    rng = _rng(3)
    N, d, scale = 50, 8, 0.5
    c = 40.0 / scale
    k = rng.standard_normal((1, N, d))
    k[0, :, 0] = 0.0
    q = rng.standard_normal((1, N, d))
    q[0, :, :] = 0.0
    q[0, :, 0] = c
    js = rng.integers(0, N)
    k[0, js, :] = 0.0
    k[0, js, 0] = 1.0
    v = rng.standard_normal((1, N, d))
    o, lse = orc.forward(q, k, v, scale, False)
    bound = N * math.exp(-40.0) * np.abs(v).max() * 2
    _close(o, np.broadcast_to(v[0, js], (N, d)), 0.0, atol=bound, what="one-hot O")
    _close(lse, np.full(N, 40.0), 0.0, atol=N * math.exp(-40.0) * 2, what="one-hot lse")
    # causal: for rows i >= j* the key j* dominates; for rows i < j*, scores are
    # all 0 (keys orthogonal to e_1) so O_i is the prefix mean
    o, lse = orc.forward(q, k, v, scale, True)
    o = o.reshape(N, d)
    for i in range(N):
        if i >= js:
            _close(o[i], v[0, js], 0.0, atol=bound, what=f"causal one-hot row {i}")
        else:
            _close(o[i], v[0, : i + 1].mean(axis=0), 1e-12, atol=1e-14,
                   what=f"causal prefix row {i}")


# ---------------------------------------------------------------- pin 4
def pin_permutation(orc):
    """Jointly permuting the rows of K and V (non-causal) leaves O, lse and dQ
    unchanged and permutes dK and dV the same way."""
    rng = _rng(4)
    BH, N, d, scale = 2, 29, 16, 0.25
    q, k, v, dO = (rng.standard_normal((BH, N, d)) for _ in range(4))
    perm = rng.permutation(N)
    o1, l1 = orc.forward(q, k, v, scale, False)
    o2, l2 = orc.forward(q, k[:, perm], v[:, perm], scale, False)
    _close(o2, o1, 1e-12, atol=1e-14, what="perm O")
    _close(l2, l1, 1e-13, what="perm lse")
    dq1, dk1, dv1, _ = orc.backward(q, k, v, dO, scale, False)
    dq2, dk2, dv2, _ = orc.backward(q, k[:, perm], v[:, perm], dO, scale, False)
    _close(dq2, dq1, 1e-11, atol=1e-13, what="perm dQ")
    dk1 = dk1.reshape(BH, N, d)[:, perm].reshape(-1, d)
    dv1 = dv1.reshape(BH, N, d)[:, perm].reshape(-1, d)
    _close(dk2, dk1, 1e-11, atol=1e-13, what="perm dK")
    _close(dv2, dv1, 1e-11, atol=1e-13, what="perm dV")


# ---------------------------------------------------------------- pin 5
def _two_pass(x):
    """Textbook two-pass safe softmax of one row (the brute force)."""
    m = max(x)
    if m == -math.inf:
        return m, 0.0
    return m, sum(math.exp(t - m) for t in x)


def pin_online_equals_two_pass(orc):
    """Brute force on tiny rows: for n <= 8 and EVERY block size 1..n, the
    online (m, l) and the online O / lse equal the two-pass values, including
    rows holding -inf entries."""
    rng = _rng(5)
    for n in range(1, 9):
        for trial in range(3):
            x = list(rng.standard_normal(n) * 3)
            if trial == 1 and n > 1:  # some -inf entries, at least one finite
                for t in rng.choice(n, size=n // 2, replace=False):
                    x[int(t)] = -math.inf
            if trial == 2 and n > 2:  # -inf in the leading block
                x[0] = -math.inf
            m_ref, l_ref = _two_pass(x)
            v = rng.standard_normal((n, 3))
            p_ref = np.array([math.exp(t - m_ref) / l_ref for t in x])
            o_ref = p_ref @ v
            for block in range(1, n + 1):
                m, l = orc.online_softmax(np.array(x), block)
                assert m[-1] == m_ref, (x, block, m, m_ref)
                _close(l[-1], l_ref, 1e-13, what=f"online l n={n} block={block}")
                o, lse = orc.online_attention_row(np.array(x), v, block)
                _close(o, o_ref, 1e-12, atol=1e-14, what=f"online O n={n} block={block}")
                _close(lse, m_ref + math.log(l_ref), 1e-13, atol=1e-15,
                       what=f"online lse n={n} block={block}")
    # and the online row against the oracle's definition on a real attention row
    N, d = 8, 4
    q = rng.standard_normal((1, N, d))
    k = rng.standard_normal((1, N, d))
    v = rng.standard_normal((1, N, d))
    for causal in (False, True):
        o_def, lse_def = orc.forward(q, k, v, 0.7, causal)
        for i in range(N):
            s = 0.7 * (k[0] @ q[0, i])
            if causal:
                s[i + 1:] = -math.inf
            for block in range(1, N + 1):
                o, lse = orc.online_attention_row(s, v[0], block)
                _close(o, o_def[i], 1e-12, atol=1e-14, what=f"online vs definition row {i}")
                _close(lse, lse_def[i], 1e-13, atol=1e-15, what=f"online lse row {i}")


# ---------------------------------------------------------------- pin 6
def pin_finite_differences(orc):
    """Central differences (h = 1e-6) of L = sum(O * dO) match dQ, dK, dV on
    B=H=1, N in {1,3,5}, d in {2,4}, causal and not."""
    rng = _rng(6)
    h = 1e-6
    for N in (1, 3, 5):
        for d in (2, 4):
            for causal in (False, True):
                q, k, v, dO = (rng.standard_normal((1, N, d)) for _ in range(4))
                scale = 1.0 / math.sqrt(d)
                dq, dk, dv, _ = orc.backward(q, k, v, dO, scale, causal, nthreads=1)
                grads = {"q": dq, "k": dk, "v": dv}

                def loss(qq, kk, vv):
                    o, _ = orc.forward(qq, kk, vv, scale, causal, nthreads=1)
                    return float(np.sum(o.reshape(1, N, d) * dO))

                for name in ("q", "k", "v"):
                    fd = np.zeros((N, d))
                    for i in range(N):
                        for c in range(d):
                            args = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
                            args[name][0, i, c] += h
                            lp = loss(args["q"], args["k"], args["v"])
                            args[name][0, i, c] -= 2 * h
                            lm = loss(args["q"], args["k"], args["v"])
                            fd[i, c] = (lp - lm) / (2 * h)
                    g = grads[name].reshape(N, d)
                    err = np.linalg.norm(fd - g)
                    assert err <= 1e-7 * max(np.linalg.norm(g), 1e-2), \
                        (name, N, d, causal, err, np.linalg.norm(g))


# ---------------------------------------------------------------- pin 7
def pin_structure(orc):
    """Invariants of the definition:
    * D = sum_j P_ij dP_ij equals sum_c dO_ic O_ic (rows of dS sum to zero);
    * N = 1: O = V and lse = scale q.k;
    * O is linear in V;
    * adding c to every K row leaves O, dQ, dK, dV unchanged and shifts lse_i
      by scale q_i.c (the row-constant shift cancels in the softmax, and
      sum_j dS_ij = 0 keeps dQ fixed)."""
    rng = _rng(7)
    BH, N, d, scale = 2, 23, 8, 0.35
    q, k, v, dO = (rng.standard_normal((BH, N, d)) for _ in range(4))
    for causal in (False, True):
        dq, m, l, D, D_alt = orc.backward_rows(q, k, v, dO, scale, causal)
        _close(D, D_alt, 1e-12, atol=1e-13, what="D two ways")
        o, lse = orc.forward(q, k, v, scale, causal)
        _close(m + np.log(l), lse, 1e-13, what="m + ln l == lse")
        _close(D, np.sum(o * dO.reshape(-1, d), axis=1), 1e-11, atol=1e-13,
               what="D == rowsum(dO*O)")
    # N = 1
    q1, k1, v1 = q[:, :1], k[:, :1], v[:, :1]
    o, lse = orc.forward(q1, k1, v1, scale, False)
    _close(o, v1.reshape(-1, d), 1e-15, what="N=1 O")
    _close(lse, scale * np.sum(q1 * k1, axis=2).reshape(-1), 1e-13, atol=1e-15, what="N=1 lse")
    # linear in V
    v2 = rng.standard_normal((BH, N, d))
    for causal in (False, True):
        oa, _ = orc.forward(q, k, v, scale, causal)
        ob, _ = orc.forward(q, k, v2, scale, causal)
        oc, _ = orc.forward(q, k, 2.0 * v - 3.0 * v2, scale, causal)
        _close(oc, 2.0 * oa - 3.0 * ob, 1e-11, atol=1e-13, what="linear in V")
    # K shift
    cvec = rng.standard_normal(d)
    for causal in (False, True):
        o1, l1 = orc.forward(q, k, v, scale, causal)
        o2, l2 = orc.forward(q, k + cvec, v, scale, causal)
        _close(o2, o1, 1e-10, atol=1e-12, what="K shift O")
        _close(l2, l1 + scale * (q.reshape(-1, d) @ cvec), 1e-12, atol=1e-13,
               what="K shift lse")
        g1 = orc.backward(q, k, v, dO, scale, causal)
        g2 = orc.backward(q, k + cvec, v, dO, scale, causal)
        for a, b, nm in zip(g2[:3], g1[:3], ("dQ", "dK", "dV")):
            _close(a, b, 1e-9, atol=1e-11, what=f"K shift {nm}")


# ---------------------------------------------------------------- pin 8
def pin_torch_sdpa(orc):
    """Cross-check against an independent implementation: PyTorch's
    scaled_dot_product_attention in fp64 on the CPU with autograd gradients,
    and torch.logsumexp for lse."""
    rng = _rng(8)
    for (B, H, N, d) in ((2, 3, 37, 16), (1, 2, 130, 8)):
        for causal in (False, True):
            q, k, v, dO = (rng.standard_normal((B, H, N, d)) for _ in range(4))
            scale = 1.0 / math.sqrt(d)
            tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True)
                          for a in (q, k, v))
            to = torch.nn.functional.scaled_dot_product_attention(
                tq, tk, tv, is_causal=causal, scale=scale)
            to.backward(torch.tensor(dO))
            s = (tq @ tk.transpose(-1, -2)).detach() * scale
            if causal:
                s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), -math.inf)
            tlse = torch.logsumexp(s, dim=-1).reshape(-1).numpy()
            o, lse = orc.forward(q, k, v, scale, causal)
            _close(o, to.detach().reshape(-1, d).numpy(), 1e-10, atol=1e-12, what="sdpa O")
            _close(lse, tlse, 1e-12, atol=1e-13, what="sdpa lse")
            dq, dk, dv, _ = orc.backward(q, k, v, dO, scale, causal)
            for a, t, nm in ((dq, tq, "dQ"), (dk, tk, "dK"), (dv, tv, "dV")):
                _close(a, t.grad.reshape(-1, d).numpy(), 1e-9, atol=1e-11, what=f"sdpa {nm}")


# ---------------------------------------------------------------- pin 9
def pin_selection_consistency(orc):
    """Selected-row / selected-column calls return exactly the corresponding
    rows of the full computation (the sampled checks rely on this)."""
    rng = _rng(9)
    BH, N, d, scale = 3, 41, 8, 0.3
    q, k, v, dO = (rng.standard_normal((BH, N, d)) for _ in range(4))
    rows = np.array([0, 5, N - 1, N, 2 * N + 7, BH * N - 1])
    for causal in (False, True):
        o, lse = orc.forward(q, k, v, scale, causal)
        os_, ls_ = orc.forward(q, k, v, scale, causal, rows=rows)
        assert np.array_equal(os_, o[rows]) and np.array_equal(ls_, lse[rows])
        dq, dk, dv, (m, l, D, _) = orc.backward(q, k, v, dO, scale, causal)
        dqs, *_ = orc.backward_rows(q, k, v, dO, scale, causal, rows=rows)
        dks, dvs = orc.backward_cols(q, k, v, dO, m, l, D, scale, causal, cols=rows)
        assert np.array_equal(dqs, dq[rows])
        assert np.array_equal(dks, dk[rows]) and np.array_equal(dvs, dv[rows])


# ---------------------------------------------------------------- pin 10
def _expand(mask, bq, bk, N):
    """Element mask [.., N, N] from a block mask [.., nqb, nkb]."""
    m = np.asarray(mask, dtype=bool)
    return np.repeat(np.repeat(m, bq, axis=-2), bk, axis=-1)[..., :N, :N]


def pin_block_mask(orc):
    """Block-sparse masking (the talk's block-sparse FlashAttention):
    * an all-ones block mask changes nothing (bit for bit);
    * a block-diagonal mask splits the problem into independent dense
      attention problems, one per block (O, lse and all three gradients);
    * against PyTorch's fp64 SDPA with the element-expanded boolean mask,
      with uneven block sizes (bq != bk), per-head masks and causal on top;
    * rows whose blocks are all dropped give o = 0, lse = -inf and zero dq,
      and do not change dk, dv of other rows."""
    rng = _rng(10)
    BH, N, d, scale = 2, 22, 8, 0.4
    q, k, v, dO = (rng.standard_normal((BH, N, d)) for _ in range(4))
    ones = np.ones((6, 8), np.uint8)  # bq=4, bk=3
    a = orc.forward(q, k, v, scale, True)
    b = orc.forward(q, k, v, scale, True, mask=ones, block=(4, 3))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # block diagonal with square blocks of 5 rows: independent sub-problems
    nb = -(-N // 5)
    diag = np.eye(nb, dtype=np.uint8)
    o, lse = orc.forward(q, k, v, scale, False, mask=diag, block=(5, 5))
    dq, dk, dv, _ = orc.backward(q, k, v, dO, scale, False, mask=diag, block=(5, 5))
    o, lse, dq, dk, dv = (x.reshape(BH, N, *x.shape[1:]) for x in (o, lse, dq, dk, dv))
    for b0 in range(0, N, 5):
        sl = slice(b0, min(b0 + 5, N))
        ob, lb = orc.forward(q[:, sl], k[:, sl], v[:, sl], scale, False)
        gq, gk, gv, _ = orc.backward(q[:, sl], k[:, sl], v[:, sl], dO[:, sl], scale, False)
        n = sl.stop - sl.start
        _close(o[:, sl].reshape(-1, d), ob, 1e-13, atol=1e-15, what="block-diag O")
        _close(lse[:, sl].reshape(-1), lb, 1e-13, atol=1e-15, what="block-diag lse")
        for got, ref, nm in ((dq, gq, "dQ"), (dk, gk, "dK"), (dv, gv, "dV")):
            _close(got[:, sl].reshape(-1, d), ref.reshape(BH * n, d), 1e-12, atol=1e-14,
                   what=f"block-diag {nm}")
    # random per-head masks, uneven blocks, against torch SDPA (every row keeps a block)
    bq, bk = 4, 3
    nqb, nkb = -(-N // bq), -(-N // bk)
    for causal in (False, True):
        mask = (rng.random((BH, nqb, nkb)) < 0.5).astype(np.uint8)
        mask[:, :, 0] = 1  # key block 0 is visible to every row (also under causal)
        el = _expand(mask, bq, bk, N)
        if causal:
            el = el & np.tril(np.ones((N, N), dtype=bool))
        tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
        to = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, attn_mask=torch.tensor(el), scale=scale)
        to.backward(torch.tensor(dO))
        s_ = (tq @ tk.transpose(-1, -2)).detach() * scale
        tlse = torch.logsumexp(s_.masked_fill(~torch.tensor(el), -math.inf), dim=-1)
        o, lse = orc.forward(q, k, v, scale, causal, mask=mask, block=(bq, bk))
        dq, dk, dv, _ = orc.backward(q, k, v, dO, scale, causal, mask=mask, block=(bq, bk))
        _close(o, to.detach().reshape(-1, d).numpy(), 1e-10, atol=1e-12, what="masked O vs sdpa")
        _close(lse, tlse.reshape(-1).numpy(), 1e-12, atol=1e-13, what="masked lse vs sdpa")
        for got, t, nm in ((dq, tq, "dQ"), (dk, tk, "dK"), (dv, tv, "dV")):
            _close(got, t.grad.reshape(-1, d).numpy(), 1e-9, atol=1e-11, what=f"masked {nm}")
    # fully dropped query block 1 (rows 4..7): o = 0, lse = -inf, dq = 0
    mask = np.ones((nqb, nkb), np.uint8)
    mask[1, :] = 0
    o, lse = orc.forward(q, k, v, scale, False, mask=mask, block=(bq, bk))
    dq, dk, dv, _ = orc.backward(q, k, v, dO, scale, False, mask=mask, block=(bq, bk))
    o, lse, dq = o.reshape(BH, N, d), lse.reshape(BH, N), dq.reshape(BH, N, d)
    assert np.all(o[:, 4:8] == 0.0) and np.all(lse[:, 4:8] == -np.inf) and np.all(dq[:, 4:8] == 0)
    # a dropped row contributes nothing to dK, dV: same as the unmasked problem
    # with that row's upstream gradient set to zero
    dO0 = dO.copy()
    dO0[:, 4:8] = 0.0
    g = orc.backward(q, k, v, dO0, scale, False)
    _close(dk, g[1], 1e-12, atol=1e-14, what="dK without the dropped rows")
    _close(dv, g[2], 1e-12, atol=1e-14, what="dV without the dropped rows")


# ---------------------------------------------------------------- pin 11
def pin_decode(orc):
    """Decode (a few queries against a key/value cache):
    * with Nq = Nk it is the square definition (causal alignments coincide);
    * against PyTorch's fp64 SDPA with the explicit mask "query i sees keys
      up to Nk - Nq + i", for Nq < Nk;
    * splitting the keys into two ranges and merging the two partial results
      with the running-max update (transcript 04:46-05:17: new max, the two
      rescale factors, summed and renormalised) gives the whole result;
    * one key: o = v and lse = scale q.k."""
    rng = _rng(11)
    BH, d, scale = 3, 16, 0.25
    q, k, v = (rng.standard_normal((BH, 40, d)) for _ in range(3))
    for causal in (False, True):
        a = orc.forward(q, k, v, scale, causal)
        b = orc.decode(q, k, v, scale, causal)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    Nq, Nk = 5, 37
    q = rng.standard_normal((BH, Nq, d))
    k, v = (rng.standard_normal((BH, Nk, d)) for _ in range(2))
    for causal in (False, True):
        mask = np.ones((Nq, Nk), dtype=bool)
        if causal:
            mask = np.arange(Nk)[None, :] <= (Nk - Nq + np.arange(Nq))[:, None]
        tq, tk, tv = (torch.tensor(x) for x in (q, k, v))
        to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv,
                                                             attn_mask=torch.tensor(mask),
                                                             scale=scale)
        sc = (tq @ tk.transpose(-1, -2)) * scale
        tlse = torch.logsumexp(sc.masked_fill(~torch.tensor(mask), -math.inf), dim=-1)
        o, lse = orc.decode(q, k, v, scale, causal)
        _close(o, to.reshape(-1, d).numpy(), 1e-12, atol=1e-14, what="decode O vs sdpa")
        _close(lse, tlse.reshape(-1).numpy(), 1e-13, atol=1e-14, what="decode lse vs sdpa")
    # split the cache at a = 15 and merge
    a_ = 15
    o, lse = orc.decode(q, k, v, scale, False)
    o1, l1 = orc.decode(q, k[:, :a_], v[:, :a_], scale, False)
    o2, l2 = orc.decode(q, k[:, a_:], v[:, a_:], scale, False)
    m = np.maximum(l1, l2)
    w1, w2 = np.exp(l1 - m), np.exp(l2 - m)
    merged = (w1[:, None] * o1 + w2[:, None] * o2) / (w1 + w2)[:, None]
    _close(merged, o, 1e-12, atol=1e-14, what="split-merge O")
    _close(m + np.log(w1 + w2), lse, 1e-13, atol=1e-14, what="split-merge lse")
    o, lse = orc.decode(q[:, :1], k[:, :1], v[:, :1], scale, True)
    _close(o, v[:, 0], 1e-15, what="one-key O")
    _close(lse, scale * np.sum(q[:, 0] * k[:, 0], axis=1), 1e-13, atol=1e-15, what="one-key lse")


# ---------------------------------------------------------------- pin 12
def _read_kat(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, _, val = line.partition("=")
                vals[key.strip()] = [int(w, 16) for w in val.split()]
    return vals


def _z_scores(count, n, prob):
    """How many standard deviations a binomial count is from its mean."""
    return abs(count - n * prob) / math.sqrt(n * prob * (1.0 - prob))


def pin_dropout(orc):
    """Dropout on P (O = (P o Z / q) V with q the keep probability, lse that
    of P), with Z replayed from Philox4x32-10.

    The generator against its published known-answer vectors; p = 0 against
    the plain definition (bit for bit); the keep decisions against their
    distribution (keep rate, every bit of the word fair, independent across
    heads, offsets and seeds); the forward against the closed form it has
    when V is the identity (O is then the dropped, rescaled P); the whole
    backward against PyTorch fp64 autograd of the same expression given Z;
    and unbiasedness: averaged over seeds, O tends to the undropped O.
    """
    kat = _read_kat("philox4x32_10_kat.txt")
    for nm in ("zero", "ones", "pi"):
        got = orc.philox(kat[nm + "_ctr"], kat[nm + "_key"])
        assert got == kat[nm + "_out"], f"Philox known answer {nm}: {got}"

    rng = _rng(12)
    BH, N, d, scale = 2, 37, 8, 0.4
    q, k, v, dO = (rng.standard_normal((BH, N, d)) for _ in range(4))
    for causal in (False, True):
        o0, l0 = orc.forward(q, k, v, scale, causal)
        o1, l1 = orc.forward(q, k, v, scale, causal, dropout=(0.0, 99, 3))
        assert np.array_equal(o0, o1) and np.array_equal(l0, l1), "p = 0 changes O"
        g0 = orc.backward(q, k, v, dO, scale, causal)
        g1 = orc.backward(q, k, v, dO, scale, causal, dropout=(0.0, 99, 3))
        for a, b in zip(g0[:3], g1[:3]):
            assert np.array_equal(a, b), "p = 0 changes a gradient"

    # keep decisions: the 16-bit values are the halves of the generator's
    # words; rate, fair bits, independence
    p, seed, off = 0.2, 0x1234_5678_9ABC_DEF0, 7
    rows, cols = 48, 256
    u16 = np.array([[orc.dropout_u16(seed, off, 1, i, j) for j in range(cols)]
                    for i in range(rows)], dtype=np.uint64)
    words = orc.philox([0, 5, 1, off], [seed & 0xFFFFFFFF, seed >> 32])
    assert [int(u16[5, 2 * e]) | (int(u16[5, 2 * e + 1]) << 16) for e in range(4)] == words
    n = u16.size
    keep = orc.dropout_keep(p, seed, off, 1, rows, cols)
    thr, rs = oracle_dropout_params(p)
    assert thr == int(np.floor(float(np.float32(p)) * 65536)) and rs == 65536 / (65536 - thr)
    assert np.array_equal(keep, u16 >= thr)
    assert _z_scores(int(keep.sum()), n, 1.0 - thr / 65536) < 5.0, "keep rate"
    for b in range(16):
        assert _z_scores(int(((u16 >> b) & 1).sum()), n, 0.5) < 5.0, f"bit {b} biased"
    for other in ((seed, off, 0), (seed, off + 1, 1), (seed ^ 1, off, 1), (seed ^ 2**40, off, 1)):
        keep2 = np.array([[orc.dropout_u16(other[0], other[1], other[2], i, j) >= thr
                           for j in range(cols)] for i in range(rows)])
        agree = int((keep == keep2).sum())
        assert _z_scores(agree, n, p * p + (1 - p) * (1 - p)) < 5.0, f"not independent {other}"

    # V = identity: O_ij = P_ij Z_ij / q exactly
    Nn = 24
    qq, kk = rng.standard_normal((2, Nn, Nn)), rng.standard_normal((2, Nn, Nn))
    eye = np.broadcast_to(np.eye(Nn), (2, Nn, Nn)).copy()
    P, _ = orc.forward(qq, kk, eye, 0.3, False)
    pd, seed2, off2 = 0.35, 2024, 5
    O, _ = orc.forward(qq, kk, eye, 0.3, False, dropout=(pd, seed2, off2))
    _, rs = oracle_dropout_params(pd)
    for bh in range(2):
        Z = orc.dropout_keep(pd, seed2, off2, bh, Nn, Nn)
        _close(O[bh * Nn:(bh + 1) * Nn], P[bh * Nn:(bh + 1) * Nn] * Z * rs, 1e-15,
               what="dropout closed form")

    # backward against autograd of the same expression given Z
    pd, seed3, off3 = 0.25, 77, 1
    _, rs = oracle_dropout_params(pd)
    Z = np.stack([orc.dropout_keep(pd, seed3, off3, bh, N, N) for bh in range(BH)])
    for causal in (False, True):
        tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
        s_ = (tq @ tk.transpose(-1, -2)) * scale
        if causal:
            s_ = s_.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), -math.inf)
        to = (torch.softmax(s_, dim=-1) * torch.tensor(Z, dtype=torch.float64) * rs) @ tv
        to.backward(torch.tensor(dO))
        o, lse = orc.forward(q, k, v, scale, causal, dropout=(pd, seed3, off3))
        _close(o, to.detach().reshape(-1, d).numpy(), 1e-10, atol=1e-12, what="dropout O")
        _close(lse, torch.logsumexp(s_.detach(), -1).reshape(-1).numpy(), 1e-12, atol=1e-13,
               what="dropout lse")
        dq, dk, dv, (_, _, D, D_alt) = orc.backward(q, k, v, dO, scale, causal,
                                                    dropout=(pd, seed3, off3))
        _close(D, D_alt, 1e-10, atol=1e-12, what="dropout D forms")
        for a, t, nm in ((dq, tq, "dQ"), (dk, tk, "dK"), (dv, tv, "dV")):
            _close(a, t.grad.reshape(-1, d).numpy(), 1e-9, atol=1e-11, what=f"dropout {nm}")

    # unbiased: E[O] over seeds is the undropped O
    Bs, Ns, ds = 1, 12, 4
    q4, k4, v4 = (rng.standard_normal((Bs, Ns, ds)) for _ in range(3))
    ref, _ = orc.forward(q4, k4, v4, 0.5, False)
    samples = np.stack([orc.forward(q4, k4, v4, 0.5, False, dropout=(0.3, s4, 0), nthreads=1)[0]
                        for s4 in range(600)])
    se = samples.std(axis=0) / math.sqrt(samples.shape[0])
    assert np.all(np.abs(samples.mean(axis=0) - ref) <= 5.0 * se + 1e-12), "dropout biased"


ALL_PINS = [pin_worked_example, pin_zero_query, pin_one_hot, pin_permutation,
            pin_online_equals_two_pass, pin_finite_differences, pin_structure,
            pin_torch_sdpa, pin_selection_consistency, pin_block_mask, pin_decode,
            pin_dropout]
