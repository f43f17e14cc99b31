"""Pins of the fp64 CPU oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle (oracle/path_oracle.c) against something other than itself:
explicit d x d matrix products, library softmax attention, worked examples printed on the
pages (tests/golden/worked_examples.json), a closed-form permutation logit, the linear-RNN
recurrence, the UT / blockwise identities written out from the pages, and finite differences.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def rand_problem(rng, L, d, beta_lo=0.0, beta_hi=2.0, fox=False):
    q = rng.standard_normal((L, d))
    k = rng.standard_normal((L, d))
    v = rng.standard_normal((L, d))
    w = rng.standard_normal((L, d))
    w /= np.linalg.norm(w, axis=-1, keepdims=True)
    beta = rng.uniform(beta_lo, beta_hi, L)
    logf = np.log(1.0 / (1.0 + np.exp(-(rng.standard_normal(L) + 2.0)))) if fox else None
    return q, k, v, w, beta, logf


def explicit_logits(q, k, w, beta, logf, scale):
    """Brute force: S_ij = scale k_j^T (H_{j+1} @ ... @ H_i) q_i + sum_{s=j+1..i} log f_s."""
    L, d = q.shape
    H = [np.eye(d) - beta[t] * np.outer(w[t], w[t]) for t in range(L)]
    S = np.full((L, L), -np.inf)
    for i in range(L):
        for j in range(i + 1):
            F = np.eye(d)
            for t in range(j + 1, i + 1):
                F = F @ H[t]
            bias = 0.0 if logf is None else float(sum(logf[j + 1:i + 1]))
            S[i, j] = scale * k[j] @ F @ q[i] + bias
    return S


def softmax_attend(S, v):
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    P /= P.sum(axis=1, keepdims=True)
    lse = (m[:, 0] + np.log(np.exp(S - m).sum(axis=1)))
    return P @ v, lse


@pytest.mark.parametrize("L,d,fox,scale", [(1, 3, False, 1.0), (7, 4, False, 0.7), (12, 8, True, 1.3),
                                           (11, 5, True, 2.0), (9, 128, True, 1.0)])
def test_logits_and_outputs_match_explicit_products(L, d, fox, scale):
    rng = np.random.default_rng(L * 100 + d)
    q, k, v, w, beta, logf = rand_problem(rng, L, d, fox=fox)
    S_ref = explicit_logits(q, k, w, beta, logf, scale)
    S = orc.logits(q, k, w, beta, logf, scale)
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-12)
    o_ref, lse_ref = softmax_attend(S_ref, v)
    o, lse = orc.fwd(q[None], k[None], v[None], w[None], beta[None],
                     None if logf is None else logf[None], scale)
    np.testing.assert_allclose(o[0], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0], lse_ref, rtol=0, atol=1e-12)


def test_path_endpoints():
    """H_j is outside the path of key j, H_i inside the path of query i (notes §2.1)."""
    d, L = 3, 2
    q = np.array([[0, 0, 0], [1.0, 2.0, 3.0]])
    k = np.array([[1.0, 0, 0], [0, 0, 0]])
    w = np.array([[0, 1.0, 0], [1.0, 0, 0]])
    # H_0 erases e2 (must NOT act); H_1 flips e1 (MUST act on q_1 before scoring k_0)
    beta = np.array([1.0, 2.0])
    S = orc.logits(q, k, w, beta, None, 1.0)
    assert S[1, 0] == pytest.approx(-1.0, abs=1e-15)
    assert S[1, 1] == pytest.approx(0.0, abs=1e-15)


@pytest.mark.parametrize("scale", [1.0, 0.125, 16.0])
def test_beta_zero_is_causal_softmax_attention(scale):
    rng = np.random.default_rng(3)
    n, L, d = 3, 40, 16
    q, k, v = (rng.standard_normal((n, L, d)) / 4 for _ in range(3))
    w = rng.standard_normal((n, L, d))
    w /= np.linalg.norm(w, axis=-1, keepdims=True)
    beta = np.zeros((n, L))
    o, lse = orc.fwd(q, k, v, w, beta, None, scale)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q), torch.tensor(k), torch.tensor(v), is_causal=True, scale=scale).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    S = scale * np.einsum("nid,njd->nij", q, k) + np.triu(np.full((L, L), -np.inf), 1)
    lse_ref = torch.logsumexp(torch.tensor(S), dim=-1).numpy()
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def _transported_queries(q, w, beta):
    """z_{i,j} = H_{j+1}..H_i q_i read back coordinate by coordinate through the oracle's
    logits, using keys equal to the standard basis vector e_m at every position."""
    L, d = q.shape
    Z = np.zeros((L, L, d))
    for m in range(d):
        k = np.zeros((L, d))
        k[:, m] = 1.0
        S = orc.logits(q, k, w, beta, None, 1.0)
        Z[:, :, m] = np.where(np.isfinite(S), S, 0.0)
    return Z


def test_out_of_range_beta_is_clamped_to_the_parameterisation_range():
    """beta = 2 sigmoid(x) lives in (0, 2) (notes §2.1); values outside are read as clamped to
    [0, 2].  Logits and outputs at beta = -0.5 / 2.5 are the explicit products at beta = 0 / 2 (and
    differ from the unclamped products), and every gradient, dbeta included, is the one at the
    clamped value."""
    rng = np.random.default_rng(31)
    L, d = 10, 6
    q, k, v, w, beta, _ = rand_problem(rng, L, d)
    beta[[1, 4, 8]] = [-0.5, 2.5, 2.5]
    clamped = np.clip(beta, 0.0, 2.0)
    assert clamped[1] == 0.0 and clamped[4] == 2.0
    S = orc.logits(q, k, w, beta, None, 1.0)
    np.testing.assert_allclose(S, explicit_logits(q, k, w, clamped, None, 1.0), rtol=0, atol=1e-12)
    low = np.tril_indices(L)
    assert np.abs(S[low] - explicit_logits(q, k, w, beta, None, 1.0)[low]).max() > 1e-3
    o, lse = orc.fwd(q[None], k[None], v[None], w[None], beta[None], None, 1.0)
    o_ref, lse_ref = softmax_attend(explicit_logits(q, k, w, clamped, None, 1.0), v)
    np.testing.assert_allclose(o[0], o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0], lse_ref, rtol=0, atol=1e-12)
    dO = rng.standard_normal((L, d))
    g_out = orc.bwd(q[None], k[None], v[None], w[None], beta[None], None, 1.0, dO[None])
    g_in = orc.bwd(q[None], k[None], v[None], w[None], clamped[None], None, 1.0, dO[None])
    for key in ("dq", "dk", "dv", "dw", "dbeta"):
        np.testing.assert_allclose(g_out[key], g_in[key], rtol=0, atol=1e-12, err_msg=key)


def test_beta_two_preserves_norm_and_smaller_beta_contracts():
    rng = np.random.default_rng(5)
    L, d = 10, 6
    q, _, _, w, _, _ = rand_problem(rng, L, d)
    Z = _transported_queries(q, w, np.full(L, 2.0))
    qn = np.linalg.norm(q, axis=-1)
    for i in range(L):
        for j in range(i + 1):
            assert np.linalg.norm(Z[i, j]) == pytest.approx(qn[i], rel=1e-12)
    Z2 = _transported_queries(q, w, np.full(L, 1.5))
    # every H with beta in (0,2) is a contraction: norms never increase along the walk
    for i in range(L):
        norms = [np.linalg.norm(Z2[i, j]) for j in range(i, -1, -1)]
        assert all(b <= a * (1 + 1e-12) for a, b in zip(norms, norms[1:]))
        if i >= 2:
            assert norms[-1] < qn[i] * (1 - 1e-6)


@pytest.mark.parametrize("name", ["swap", "erase"])
def test_worked_examples_from_the_notes(name):
    ex = GOLDEN[name]
    w1 = np.array(ex["w"])
    d = len(w1)
    H = np.zeros((d, d))
    for m in range(d):
        for n in range(d):
            # position 0: key e_m; position 1: transition (w1, beta) and query e_n
            q = np.zeros((2, d)); q[1, n] = 1.0
            k = np.zeros((2, d)); k[0, m] = 1.0
            w = np.stack([np.eye(d)[0], w1])
            beta = np.array([0.0, ex["beta"]])
            H[m, n] = orc.logits(q, k, w, beta, None, 1.0)[1, 0]
    np.testing.assert_allclose(H, np.array(ex["H"]), rtol=0, atol=1e-15)


def test_eigenstructure_of_one_transition():
    """H z = z_perp + (1 - beta) alpha w (notes §2.2), read through a one-step path."""
    rng = np.random.default_rng(11)
    d = 5
    w1 = rng.standard_normal(d); w1 /= np.linalg.norm(w1)
    perp = rng.standard_normal(d); perp -= (perp @ w1) * w1
    for beta1 in GOLDEN["eigen"]["beta_values"]:
        for alpha in (0.3, -1.7):
            zq = perp + alpha * w1
            expect = perp + (1 - beta1) * alpha * w1
            got = np.zeros(d)
            for m in range(d):
                q = np.stack([np.zeros(d), zq]); k = np.zeros((2, d)); k[0, m] = 1.0
                w = np.stack([w1, w1])
                got[m] = orc.logits(q, k, w, np.array([0.0, beta1]), None, 1.0)[1, 0]
            np.testing.assert_allclose(got, expect, rtol=0, atol=1e-14)


def _transposition_w(a, b, d):
    w = np.zeros(d)
    w[a], w[b] = 1 / math.sqrt(2), -1 / math.sqrt(2)
    return w


def test_theorem21_permutation_logit():
    th = GOLDEN["theorem21"]
    n5 = th["n_elements"]
    base = np.arange(1, n5 + 1, dtype=float)
    # the page's numbers: identity gives 55, every other permutation at most 54
    sums = {p: sum((r + 1) * (p[r] + 1) for r in range(n5)) for p in itertools.permutations(range(n5))}
    assert sums[tuple(range(n5))] == th["identity_sum"]
    assert max(s for p, s in sums.items() if p != tuple(range(n5))) == th["max_non_identity_sum"]

    rng = np.random.default_rng(21)
    d = 8  # five used coordinates, padded
    for trial in range(30):
        nsw = int(rng.integers(1, 12))
        pairs = [tuple(rng.choice(n5, 2, replace=False)) for _ in range(nsw)]
        if trial % 3 == 0:  # force an identity composition: a sequence followed by its reverse
            pairs = pairs + pairs[::-1]
        L = len(pairs) + 2
        q = np.zeros((L, d)); k = np.zeros((L, d)); w = np.zeros((L, d)); beta = np.zeros(L)
        k[0, :n5] = base
        q[-1, :n5] = base
        w[0, 0] = 1.0
        w[-1, 0] = 1.0
        for t, (a, b) in enumerate(pairs, start=1):
            w[t] = _transposition_w(a, b, d)
            beta[t] = 2.0
        s = orc.logits(q, k, w, beta, None, 1.0)[L - 1, 0]
        # integer composition: apply T_n first, ..., T_1 last to the vector (1..5)
        vec = list(range(1, n5 + 1))
        for a, b in reversed(pairs):
            vec[a], vec[b] = vec[b], vec[a]
        expect = sum((r + 1) * vec[r] for r in range(n5))
        assert s == pytest.approx(expect, abs=1e-12)
        is_identity = vec == list(range(1, n5 + 1))
        nlen = L
        s0 = nlen * (s - th["offset"])
        if is_identity:
            assert s0 == pytest.approx(nlen / 2, abs=1e-9)
        else:
            assert s0 <= -nlen / 2 + 1e-9


def test_linear_rnn_recurrence_gives_the_logits():
    """S_t = S_{t-1} H_t + v_t k_t^T, o_t = S_t q_t (notes §2.3): with one-hot values the
    coefficient of v_j in o_t is the PaTH logit (t, j)."""
    rng = np.random.default_rng(7)
    L, d = 9, 5
    q, k, _, w, beta, _ = rand_problem(rng, L, d)
    S_or = orc.logits(q, k, w, beta, None, 1.0)
    state = np.zeros((L, d))
    for t in range(L):
        H = np.eye(d) - beta[t] * np.outer(w[t], w[t])
        state = state @ H + np.outer(np.eye(L)[t], k[t])
        c = state @ q[t]
        np.testing.assert_allclose(c[:t + 1], S_or[t, :t + 1], rtol=0, atol=1e-12)
        np.testing.assert_allclose(c[t + 1:], 0.0, atol=0)


def ut_factor(W, beta):
    """U = (I + strictLower(D W W^T))^{-1} D (notes §2.6), solved by forward substitution."""
    n = W.shape[0]
    G = W @ W.T
    U = np.zeros((n, n))
    for i in range(n):
        row = np.zeros(n); row[i] = 1.0
        for kk in range(i):
            row -= G[i, kk] * U[kk]
        U[i] = beta[i] * row
    return U


def test_ut_products_and_full_matrix_form():
    rng = np.random.default_rng(9)
    L, d = 12, 5
    q, k, _, w, beta, _ = rand_problem(rng, L, d)
    U = ut_factor(w, beta)
    H = [np.eye(d) - beta[t] * np.outer(w[t], w[t]) for t in range(L)]
    left = np.eye(d)
    for t in range(L):
        left = H[t] @ left  # H_L ... H_1
    right = np.eye(d)
    for t in range(L):
        right = right @ H[t]  # H_1 ... H_L
    np.testing.assert_allclose(left, np.eye(d) - w.T @ U @ w, atol=1e-12)
    np.testing.assert_allclose(right, np.eye(d) - w.T @ U.T @ w, atol=1e-12)
    At = np.tril(q @ k.T) - np.tril(q @ w.T) @ U @ np.tril(w @ k.T, -1)
    S = orc.logits(q, k, w, beta, None, 1.0)
    np.testing.assert_allclose(np.tril(At), np.where(np.isfinite(S), S, 0.0), atol=1e-12)


@pytest.mark.parametrize("B", [1, 3, 4, 5])
def test_blockwise_right_to_left_scan(B):
    """Boundary-adjusted Q/K, chunk transforms and the right-to-left scan (notes §2.7)
    reproduce every logit of the definition, including a ragged last chunk."""
    rng = np.random.default_rng(17 + B)
    L, d = 14, 5
    q, k, _, w, beta, logf = rand_problem(rng, L, d, fox=True)
    S_or = orc.logits(q, k, w, beta, logf, 1.0)
    nc = (L + B - 1) // B
    Ql, Kr, F, Sd = [], [], [], []
    G = np.concatenate([[0.0], np.cumsum(logf)])  # prefix sums for the bias check
    for c in range(nc):
        sl = slice(c * B, min(L, (c + 1) * B))
        Wb, Qb, Kb = w[sl], q[sl], k[sl]
        U = ut_factor(Wb, beta[sl])
        X = U @ np.tril(Wb @ Kb.T, -1)
        Ql.append(Qb - np.tril(Qb @ Wb.T) @ U @ Wb)
        Kr.append(Kb - X.T @ Wb)
        F.append(np.eye(d) - Wb.T @ U.T @ Wb)
        Sd.append(np.tril(Qb @ Kb.T) - np.tril(Qb @ Wb.T) @ X)
    S = np.full((L, L), -np.inf)
    for b in range(nc):
        rows = range(b * B, min(L, (b + 1) * B))
        for a, i in enumerate(rows):
            for bb, j in enumerate(rows):
                if j <= i:
                    S[i, j] = Sd[b][a, bb] + G[i + 1] - G[j + 1]
        Z = Ql[b].copy()
        for c in range(b - 1, -1, -1):
            blk = Z @ Kr[c].T
            for a, i in enumerate(rows):
                for bb in range(blk.shape[1]):
                    j = c * B + bb
                    S[i, j] = blk[a, bb] + G[i + 1] - G[j + 1]
            Z = Z @ F[c].T
    np.testing.assert_allclose(np.where(np.isfinite(S), S, 0), np.where(np.isfinite(S_or), S_or, 0),
                               atol=1e-12)
    assert np.array_equal(np.isfinite(S), np.isfinite(S_or))


def test_decode_from_empty_cache_reproduces_forward_rows():
    """Rewriting cached keys with each new H_t (notes §2.8, Eq. (1)) gives the same outputs as
    the query walk of the forward definition."""
    rng = np.random.default_rng(13)
    n, L, d = 2, 17, 6
    q, k, v = (rng.standard_normal((n, L, d)) for _ in range(3))
    w = rng.standard_normal((n, L, d)); w /= np.linalg.norm(w, axis=-1, keepdims=True)
    beta = rng.uniform(0, 2, (n, L))
    o_f, lse_f = orc.fwd(q, k, v, w, beta, None, 0.9)
    kc = np.zeros((n, L, d)); vc = np.zeros((n, L, d))
    for t in range(L):
        o_t, lse_t = orc.decode_step(kc, vc, t, q[:, t], k[:, t], v[:, t], w[:, t], beta[:, t], 0.9,
                                     want_lse=True)
        np.testing.assert_allclose(o_t, o_f[:, t], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse_t, lse_f[:, t], rtol=0, atol=1e-12)


def test_forget_gate_special_cases():
    rng = np.random.default_rng(19)
    n, L, d = 2, 30, 8
    q, k, v = (rng.standard_normal((n, L, d)) / 3 for _ in range(3))
    w = rng.standard_normal((n, L, d)); w /= np.linalg.norm(w, axis=-1, keepdims=True)
    logf = np.log(1 / (1 + np.exp(-(rng.standard_normal((n, L)) + 2))))
    # beta = 0: bias-only attention, sum_{s=j+1..i} log f_s as an additive mask (notes §2.5)
    beta0 = np.zeros((n, L))
    o, _ = orc.fwd(q, k, v, w, beta0, logf, 1.0)
    mask = np.zeros((n, L, L))
    for h in range(n):
        for i in range(L):
            for j in range(L):
                mask[h, i, j] = logf[h, j + 1:i + 1].sum() if j <= i else -np.inf
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q), torch.tensor(k), torch.tensor(v), attn_mask=torch.tensor(mask), scale=1.0).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    # log f = 0: plain PaTH
    beta = rng.uniform(0, 2, (n, L))
    o1, l1 = orc.fwd(q, k, v, w, beta, np.zeros((n, L)), 1.0)
    o2, l2 = orc.fwd(q, k, v, w, beta, None, 1.0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def _loss(q, k, v, w, beta, logf, scale, dO):
    o, _ = orc.fwd(q[None], k[None], v[None], w[None], beta[None],
                   None if logf is None else logf[None], scale)
    return float((o[0] * dO).sum())


@pytest.mark.parametrize("fox,L,d", [(False, 9, 4), (True, 9, 4), (True, 5, 128)])
def test_gradients_match_central_differences(fox, L, d):
    rng = np.random.default_rng(23 + fox + d)
    scale = 1.3
    q, k, v, w, beta, logf = rand_problem(rng, L, d, beta_lo=0.2, beta_hi=1.8, fox=fox)
    dO = rng.standard_normal((L, d))
    g = orc.bwd(q[None], k[None], v[None], w[None], beta[None], None if logf is None else logf[None],
                scale, dO[None], want_dlogf=fox)
    params = {"q": q, "k": k, "v": v, "w": w, "beta": beta}
    grads = {"q": g["dq"][0], "k": g["dk"][0], "v": g["dv"][0], "w": g["dw"][0], "beta": g["dbeta"][0]}
    if fox:
        params["logf"] = logf
        grads["logf"] = g["dlog_f"][0]
    h = 1e-6
    for name, arr in params.items():
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            fp = _loss(q, k, v, w, beta, logf, scale, dO)
            arr[idx] = old - h
            fm = _loss(q, k, v, w, beta, logf, scale, dO)
            arr[idx] = old
            fd[idx] = (fp - fm) / (2 * h)
        err = np.abs(fd - grads[name]).max() / max(1.0, np.abs(fd).max())
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("L,d", [(16, 8), (7, 128)])
def test_gradients_match_autograd_of_explicit_products(L, d):
    """Reverse mode of an independent brute-force PyTorch fp64 formulation (explicit H matrices)."""
    rng = np.random.default_rng(29 + d)
    scale = 0.8
    q, k, v, w, beta, logf = rand_problem(rng, L, d, fox=True)
    dO = rng.standard_normal((L, d))
    T = {n: torch.tensor(a, requires_grad=True) for n, a in
         dict(q=q, k=k, v=v, w=w, beta=beta, logf=logf).items()}
    eye = torch.eye(d, dtype=torch.float64)
    H = [eye - T["beta"][t] * torch.outer(T["w"][t], T["w"][t]) for t in range(L)]
    rows = []
    for i in range(L):
        s = []
        for j in range(i + 1):
            F = eye
            for t in range(j + 1, i + 1):
                F = F @ H[t]
            s.append(scale * T["k"][j] @ F @ T["q"][i] + T["logf"][j + 1:i + 1].sum())
        p = torch.softmax(torch.stack(s), 0)
        rows.append(p @ T["v"][:i + 1])
    (torch.stack(rows) * torch.tensor(dO)).sum().backward()
    g = orc.bwd(q[None], k[None], v[None], w[None], beta[None], logf[None], scale, dO[None], want_dlogf=True)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("w", "dw"), ("beta", "dbeta"), ("logf", "dlog_f")):
        np.testing.assert_allclose(g[key][0], T[name].grad.numpy(), rtol=0, atol=1e-11, err_msg=name)


def test_fwd_rows_subset_matches_full():
    rng = np.random.default_rng(31)
    L, d = 50, 8
    q, k, v, w, beta, logf = rand_problem(rng, L, d, fox=True)
    o, lse = orc.fwd(q[None], k[None], v[None], w[None], beta[None], logf[None], 1.0)
    rows = [0, 7, 49, 23]
    o_r, lse_r = orc.fwd_rows(q, k, v, w, beta, logf, 1.0, rows)
    np.testing.assert_array_equal(o_r, o[0, rows])
    np.testing.assert_array_equal(lse_r, lse[0, rows])


# ---------------- prefill -> decode hand-off (notes §2.8, last paragraph) ----------------

def test_prefill_cache_rows_are_explicit_suffix_products():
    """Row j of the handed-off cache is H_{L-1} @ ... @ H_{j+1} k_j, formed as d x d matrices."""
    rng = np.random.default_rng(41)
    n, L, d = 2, 7, 5
    probs = [rand_problem(rng, L, d) for _ in range(n)]
    k = np.stack([p[1] for p in probs]); v = np.stack([p[2] for p in probs])
    w = np.stack([p[3] for p in probs]); beta = np.stack([p[4] for p in probs])
    kc, vc = orc.prefill_cache(k, v, w, beta, cap=L + 3)
    for h in range(n):
        for j in range(L):
            M = np.eye(d)
            for t in range(j + 1, L):  # H_t multiplies from the left: H_{L-1} ... H_{j+1}
                M = (np.eye(d) - beta[h, t] * np.outer(w[h, t], w[h, t])) @ M
            np.testing.assert_allclose(kc[h, j], M @ k[h, j], rtol=0, atol=1e-12)
        np.testing.assert_array_equal(vc[h, :L], v[h])
        assert not kc[h, L:].any() and not vc[h, L:].any()


def test_prefill_then_decode_step_gives_the_forward_row():
    """Hand off a prompt of L tokens, decode token L: o_L equals row L of the forward over L+1
    tokens (the forward oracle evaluates the path logits directly)."""
    rng = np.random.default_rng(42)
    L, d = 23, 8
    q, k, v, w, beta, _ = rand_problem(rng, L + 1, d)
    kc, vc = orc.prefill_cache(k[None, :L], v[None, :L], w[None, :L], beta[None, :L], cap=L + 1)
    o_dec = orc.decode_step(kc, vc, L, q[None, L], k[None, L], v[None, L], w[None, L], beta[None, L], scale=0.7)
    o_fwd, _ = orc.fwd(q[None], k[None], v[None], w[None], beta[None], None, 0.7)
    np.testing.assert_allclose(o_dec[0], o_fwd[0, L], rtol=0, atol=1e-12)


def test_prefill_special_cases():
    """beta = 0 leaves the keys as given; beta = 2 with w = e_0 reflects coordinate 0 once per
    later token: row j gets (-1)^(L-1-j) on that coordinate and nothing else changes."""
    rng = np.random.default_rng(43)
    L, d = 9, 4
    k = rng.standard_normal((1, L, d)); v = rng.standard_normal((1, L, d))
    w = np.zeros((1, L, d)); w[..., 0] = 1.0
    kc, _ = orc.prefill_cache(k, v, w, np.zeros((1, L)), cap=L)
    np.testing.assert_array_equal(kc[0], k[0])
    kc, _ = orc.prefill_cache(k, v, w, np.full((1, L), 2.0), cap=L)
    sign = np.array([(-1.0) ** (L - 1 - j) for j in range(L)])
    np.testing.assert_allclose(kc[0, :, 0], sign * k[0, :, 0], rtol=0, atol=1e-15)
    np.testing.assert_array_equal(kc[0, :, 1:], k[0, :, 1:])


def test_transport_keys_are_the_prefill_rows():
    """The row-at-a-time hand-off (used on full-size prompts) equals the prefill cache rows."""
    rng = np.random.default_rng(44)
    n, L, d = 3, 40, 6
    probs = [rand_problem(rng, L, d) for _ in range(n)]
    k = np.stack([p[1] for p in probs]); v = np.stack([p[2] for p in probs])
    w = np.stack([p[3] for p in probs]); beta = np.stack([p[4] for p in probs])
    kc, _ = orc.prefill_cache(k, v, w, beta, cap=L)
    rows = [0, 1, 17, 38, 39]
    np.testing.assert_allclose(orc.transport_keys(k, w, beta, rows), kc[:, rows], rtol=0, atol=1e-13)


def test_fox_decode_from_empty_cache_reproduces_forward_rows():
    """PaTH-FoX decode (key rewrite plus the forget bias carried as prefix sums) gives the FoX
    forward's rows (whose bias the forward oracle sums along the query walk)."""
    rng = np.random.default_rng(17)
    n, L, d = 2, 19, 6
    q, k, v = (rng.standard_normal((n, L, d)) for _ in range(3))
    w = rng.standard_normal((n, L, d)); w /= np.linalg.norm(w, axis=-1, keepdims=True)
    beta = rng.uniform(0, 2, (n, L))
    logf = np.log(1.0 / (1.0 + np.exp(-(rng.standard_normal((n, L)) + 2.0))))
    o_f, lse_f = orc.fwd(q, k, v, w, beta, logf, 0.9)
    kc = np.zeros((n, L, d)); vc = np.zeros((n, L, d)); ac = np.zeros((n, L))
    for t in range(L):
        o_t, lse_t = orc.decode_step_fox(kc, vc, ac, t, q[:, t], k[:, t], v[:, t], w[:, t], beta[:, t], logf[:, t],
                                         0.9, want_lse=True)
        np.testing.assert_allclose(o_t, o_f[:, t], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse_t, lse_f[:, t], rtol=0, atol=1e-12)
    np.testing.assert_allclose(ac, np.cumsum(logf, axis=1), rtol=0, atol=1e-12)


def test_fox_decode_with_zero_log_f_is_plain_decode():
    rng = np.random.default_rng(18)
    n, t0, d = 2, 9, 5
    kc = rng.standard_normal((n, t0 + 1, d)); vc = rng.standard_normal((n, t0 + 1, d))
    kc2, vc2, ac = kc.copy(), vc.copy(), np.zeros((n, t0 + 1))
    q, k, v = (rng.standard_normal((n, d)) for _ in range(3))
    w = rng.standard_normal((n, d)); w /= np.linalg.norm(w, axis=-1, keepdims=True)
    beta = rng.uniform(0, 2, n)
    o1 = orc.decode_step(kc, vc, t0, q, k, v, w, beta, 1.3)
    o2 = orc.decode_step_fox(kc2, vc2, ac, t0, q, k, v, w, beta, np.zeros(n), 1.3)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-14)
