"""Pins of the fp64 oracle against facts fixed outside the oracle itself.

Each test states the passage it rests on.  Together they are chosen so that a
plausible slip anywhere in the oracle (a dropped term, a wrong scale, a
transposed index of alpha or R, a mask on the wrong index, an off-by-one in
the window) fails at least one of them; test_planted_mistakes_are_caught
checks exactly that by compiling mutated copies of the oracle.
"""
import math
import os
import re
import tempfile

import numpy as np
import pytest

import oracle
from iha_inputs import identity_mixing, first_block_contraction

RNG = np.random.default_rng(12345)
TOL_PRINTED = 5e-7   # values printed to 6 decimals


def rand_problem(rng, B, N, H, d, P):
    D = H * d
    return dict(
        X=rng.standard_normal((B, N, D)),
        W_Q=rng.standard_normal((D, H * d)) / math.sqrt(D),
        W_K=rng.standard_normal((D, H * d)) / math.sqrt(D),
        W_V=rng.standard_normal((D, H * d)) / math.sqrt(D),
        alpha_Q=rng.standard_normal((H, H, P)) / math.sqrt(H),
        alpha_K=rng.standard_normal((H, H, P)) / math.sqrt(H),
        alpha_V=rng.standard_normal((H, H, P)) / math.sqrt(H),
        R=rng.standard_normal((H, H * P)) / math.sqrt(H * P),
    )


def run(orc, p, H, d, P, **kw):
    return orc.forward(p["X"], p["W_Q"], p["W_K"], p["W_V"], p["alpha_Q"], p["alpha_K"],
                       p["alpha_V"], p["R"], H=H, d=d, P=P, **kw)


MASKS = [(0, 0), (1, 0), (2, 1), (2, 3), (2, 100)]


# ---------------------------------------------------------------------------
# Values the pages print
# ---------------------------------------------------------------------------

def check_worked_example_causal(orc, g, projection="c"):
    """"注意力机制" section 5.4, eqs. (5.13)-(5.17): IHA with H = P = 1,
    alpha = 1, R = 1 is single-head attention; weights and outputs as printed."""
    one = np.ones((1, 1, 1))
    out, w = orc.forward(g["X"][None], g["W_Q"], g["W_K"], g["W_V"], one, one, one, np.ones((1, 1)),
                         H=1, d=2, P=1, mask_mode=1, with_weights=True, projection=projection)
    np.testing.assert_allclose(w[0, 0], g["A"], atol=TOL_PRINTED, rtol=0)
    np.testing.assert_allclose(out[0], g["O"], atol=TOL_PRINTED, rtol=0)


@pytest.mark.parametrize("projection", ["c", "numpy"])
def test_worked_example_causal(golden, projection):
    check_worked_example_causal(oracle.get(), golden("causal_single_head_example.txt"), projection)


def test_worked_example_unmasked_first_row(golden):
    """"注意力机制" exercise 5.3: the example without a mask, first row."""
    g = golden("causal_single_head_example.txt")
    e = golden("unmasked_first_row_example.txt")
    one = np.ones((1, 1, 1))
    out, w = oracle.forward(g["X"][None], g["W_Q"], g["W_K"], g["W_V"], one, one, one, np.ones((1, 1)),
                            H=1, d=2, P=1, mask_mode=0, with_weights=True)
    np.testing.assert_allclose(w[0, 0, 0], e["A0"][0], atol=TOL_PRINTED, rtol=0)
    np.testing.assert_allclose(out[0, 0], e["O0"][0], atol=TOL_PRINTED, rtol=0)


def test_worked_example_through_definition_1(golden):
    """The independent MHA loop (Definition 1) on the same printed example."""
    g = golden("causal_single_head_example.txt")
    out = oracle.mha(g["X"][None], g["W_Q"], g["W_K"], g["W_V"], H=1, d=2, mask_mode=1)
    np.testing.assert_allclose(out[0], g["O"], atol=TOL_PRINTED, rtol=0)


def test_softmax_core_exact_fractions(golden):
    """"注意力机制" eq. (5.23): rows (0,0), (log3,0), (0,log3) give weights
    1/2,1/2 | 3/4,1/4 | 1/4,3/4 and the printed outputs, exactly."""
    g = golden("cross_attention_fractions.txt")
    for u, a_ref, o_ref in zip(g["U"], g["A"], g["O"]):
        a, o = oracle.softmax_read(u, [1, 1], g["V"])
        np.testing.assert_allclose(a, a_ref, atol=1e-14, rtol=0)
        np.testing.assert_allclose(o, o_ref, atol=1e-14, rtol=0)
        a, o = oracle.softmax_read(u, [1, 0], g["V"])
        np.testing.assert_allclose(o, g["O_MASK2"][0], atol=1e-14, rtol=0)
        assert a[1] == 0.0


def test_softmax_core_rejects_empty_allowed_set():
    """"注意力机制" Algorithm 5.1: a legal row with no readable key is an error."""
    with pytest.raises(RuntimeError, match="empty"):
        oracle.softmax_read([0.0, 1.0], [0, 0], np.eye(2))


def check_scale_is_head_dim(orc, g, projection="c"):
    """Algorithm 1 scales scores by 1/sqrt(d), d = D/H the head width, not
    1/sqrt(D).  Embed the printed example as head 0 of an H = 2, d = 2
    (D = 4) problem; head 0 must still give eq. (5.17)."""
    rng = np.random.default_rng(7)
    H, d, P = 2, 2, 1
    X = np.concatenate([g["X"], rng.standard_normal((3, 2))], axis=1)[None]   # [1, 3, 4]
    def embed(w0):
        W = np.zeros((4, 4))
        W[0:2, 0:2] = w0                          # head 0 reads feature dims 0-1 only
        W[:, 2:4] = rng.standard_normal((4, 2))   # head 1: anything
        return W
    WQ, WK, WV = embed(g["W_Q"]), embed(g["W_K"]), embed(g["W_V"])
    a = identity_mixing(H, P).numpy().astype(np.float64)
    R = np.eye(H)
    out = orc.forward(X, WQ, WK, WV, a, a, a, R, H=H, d=d, P=P, mask_mode=1, projection=projection)
    np.testing.assert_allclose(out[0, :, 0:2], g["O"], atol=TOL_PRINTED, rtol=0)


@pytest.mark.parametrize("projection", ["c", "numpy"])
def test_scale_is_head_dim(golden, projection):
    check_scale_is_head_dim(oracle.get(), golden("causal_single_head_example.txt"), projection)


# ---------------------------------------------------------------------------
# Theorem 2: inclusion of MHA, strictness on repeated tokens, parameter count
# ---------------------------------------------------------------------------

def check_contains_mha(orc, mask_mode, window, P, projection="c"):
    """Theorem 2 inclusion: alpha_{m,h,j} = 1(m = h), R keeps each head's first
    pseudo-block => IHA == MHA (Definition 1).  For P >= 2 the duplicated
    pseudo-tokens at one position only rescale equal terms, so the identity
    holds under the by-position mask too."""
    rng = np.random.default_rng(100 + P + 10 * mask_mode)
    B, N, H, d = 2, 9, 3, 4
    p = rand_problem(rng, B, N, H, d, P)
    a = identity_mixing(H, P).numpy().astype(np.float64)
    p.update(alpha_Q=a, alpha_K=a, alpha_V=a, R=first_block_contraction(H, P).numpy().astype(np.float64))
    got = run(orc, p, H, d, P, mask_mode=mask_mode, window=window, projection=projection)
    ref = orc.mha(p["X"], p["W_Q"], p["W_K"], p["W_V"], H=H, d=d, mask_mode=mask_mode, window=window)
    np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("projection", ["c", "numpy"])
@pytest.mark.parametrize("mask_mode,window", MASKS)
@pytest.mark.parametrize("P", [1, 2, 3])
def test_contains_mha(mask_mode, window, P, projection):
    check_contains_mha(oracle.get(), mask_mode, window, P, projection)


def repeated_token_closed_form(x, p, H, d, P):
    """Output of every position when all N tokens equal x.

    Each pseudo-token (j', t') of head h then carries the same key k_{h,j'} and
    value v_{h,j'} for every t', and every allowed set holds the same number of
    positions for each j' (the mask reads t only).  So for pseudo-query j the
    stacked softmax collapses to a P-way softmax over j':
        pbar_{h,j} = sum_{j'} softmax_{j'}(q_{h,j} . k_{h,j'} / sqrt(d)) v_{h,j'},
    independent of t, N and the mask; then O_h = sum_{h',j} R[h, h'P+j] pbar_{h',j}.
    """
    def mixed(W, alpha):
        base = np.stack([x @ W[:, m * d:(m + 1) * d] for m in range(H)])     # [m, d]
        return np.einsum("mhj,mc->hjc", alpha, base)                            # [h, j, d]
    q, k, v = mixed(p["W_Q"], p["alpha_Q"]), mixed(p["W_K"], p["alpha_K"]), mixed(p["W_V"], p["alpha_V"])
    pbar = np.zeros((H, P, d))
    for h in range(H):
        for j in range(P):
            logits = np.array([q[h, j] @ k[h, j2] for j2 in range(P)]) / math.sqrt(d)
            w = np.exp(logits - logits.max())
            w /= w.sum()
            pbar[h, j] = w @ v[h]
    O = np.zeros((H, d))
    for h in range(H):
        for h2 in range(H):
            for j in range(P):
                O[h] += p["R"][h, h2 * P + j] * pbar[h2, j]
    return O.reshape(-1)


def check_repeated_tokens(orc, mask_mode, window, P, projection="c"):
    """Theorem 2 strictness setting (repeated-token subspace X = 1 x^T) with
    general alpha and R: the oracle must equal the closed form above."""
    rng = np.random.default_rng(200 + P + 10 * mask_mode)
    B, N, H, d = 1, 7, 3, 4
    p = rand_problem(rng, B, N, H, d, P)
    x = rng.standard_normal(H * d)
    p["X"] = np.tile(x, (B, N, 1))
    got = run(orc, p, H, d, P, mask_mode=mask_mode, window=window, projection=projection)
    ref = repeated_token_closed_form(x, p, H, d, P)
    for t in range(N):
        np.testing.assert_allclose(got[0, t], ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("projection", ["c", "numpy"])
@pytest.mark.parametrize("mask_mode,window", MASKS)
@pytest.mark.parametrize("P", [1, 2, 3])
def test_repeated_tokens_closed_form(mask_mode, window, P, projection):
    check_repeated_tokens(oracle.get(), mask_mode, window, P, projection)


def test_repeated_tokens_uniform_softmax():
    """The literal reading of the repeated-token check: when alpha_K does not
    depend on j, every score in a row is equal, the softmax is uniform, and the
    output is the R contraction of the mean pseudo-value of each head."""
    rng = np.random.default_rng(300)
    B, N, H, d, P = 1, 6, 2, 3, 2
    p = rand_problem(rng, B, N, H, d, P)
    p["alpha_K"] = np.repeat(rng.standard_normal((H, H, 1)), P, axis=2)
    x = rng.standard_normal(H * d)
    p["X"] = np.tile(x, (B, N, 1))
    got = run(oracle.get(), p, H, d, P, mask_mode=1)
    base = np.stack([x @ p["W_V"][:, m * d:(m + 1) * d] for m in range(H)])
    v = np.einsum("mhj,mc->hjc", p["alpha_V"], base)
    vmean = v.mean(axis=1)                                   # [h, d]
    ref = np.zeros((H, d))
    for h in range(H):
        for h2 in range(H):
            for j in range(P):
                ref[h] += p["R"][h, h2 * P + j] * vmean[h2]
    for t in range(N):
        np.testing.assert_allclose(got[0, t], ref.reshape(-1), atol=1e-12, rtol=0)


def test_repeated_tokens_mha_is_linear_iha_is_not():
    """Theorem 2 strictness: on X = 1 x^T, MHA is linear in x; IHA with P = 2 and
    opposite-sign pseudo-queries/keys (alpha_{.,.,2} = -alpha_{.,.,1}) and
    distinct pseudo-values is not."""
    rng = np.random.default_rng(400)
    H, d, P, N = 2, 3, 2, 4
    p = rand_problem(rng, 1, N, H, d, P)
    eye = identity_mixing(H, 1).numpy()[:, :, 0].astype(np.float64)
    p["alpha_Q"] = np.stack([eye, -eye], axis=2)
    p["alpha_K"] = np.stack([eye, -eye], axis=2)
    p["alpha_V"] = np.stack([eye, 0.5 * eye], axis=2)
    x = rng.standard_normal(H * d)
    f_iha = lambda s: run(oracle.get(), dict(p, X=np.tile(s * x, (1, N, 1))), H, d, P, mask_mode=1)[0, 0]
    f_mha = lambda s: oracle.mha(np.tile(s * x, (1, N, 1)), p["W_Q"], p["W_K"], p["W_V"], H=H, d=d, mask_mode=1)[0, 0]
    np.testing.assert_allclose(f_mha(2.0), 2.0 * f_mha(1.0), atol=1e-12)
    assert np.max(np.abs(f_iha(2.0) - 2.0 * f_iha(1.0))) > 1e-3


@pytest.mark.parametrize("H,d,P", [(4, 32, 2), (16, 64, 2), (16, 128, 4), (3, 5, 7)])
def test_parameter_count(H, d, P):
    """Theorem 2: Q + 4 H^2 P parameters, Q = 3 D^2 from the three projections
    (no bias, no output projection in Algorithm 1), 3 H^2 P from alpha and
    H^2 P from R."""
    D = H * d
    assert oracle.param_count(D, H, d, P) == 3 * D * D + 4 * H * H * P


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mask_mode,window", MASKS)
def test_rows_sum_to_one(mask_mode, window):
    """"注意力机制" Algorithm 5.1 (last step): valid rows are non-negative, sum
    to one, and forbidden positions carry weight exactly zero."""
    rng = np.random.default_rng(500)
    B, N, H, d, P = 2, 6, 2, 3, 2
    p = rand_problem(rng, B, N, H, d, P)
    _, w = run(oracle.get(), p, H, d, P, mask_mode=mask_mode, window=window, with_weights=True)
    np.testing.assert_allclose(w.sum(axis=-1), 1.0, atol=1e-13)
    assert (w >= 0).all()
    for r in range(P * N):
        t = r % N
        for c in range(P * N):
            t2 = c % N
            allowed = mask_mode == 0 or (t2 <= t and (mask_mode == 1 or t - t2 < window))
            if not allowed:
                assert (w[:, :, r, c] == 0).all()


@pytest.mark.parametrize("mask_mode,window", MASKS)
def test_stacking_order_invariance(mask_mode, window):
    """"注意力机制" eq. (5.41): a permutation applied to the tokens and, in step,
    to the visibility relation permutes the output.  Stacking pseudo-tokens
    t-major (row t*P + j) instead of j-major (row j*N + t) with a mask that
    reads t only therefore leaves every unstacked output unchanged, and
    permutes the weight matrix."""
    rng = np.random.default_rng(600)
    B, N, H, d, P = 2, 7, 2, 3, 3
    p = rand_problem(rng, B, N, H, d, P)
    o0, w0 = run(oracle.get(), p, H, d, P, mask_mode=mask_mode, window=window, stack_order=0, with_weights=True)
    o1, w1 = run(oracle.get(), p, H, d, P, mask_mode=mask_mode, window=window, stack_order=1, with_weights=True)
    np.testing.assert_allclose(o0, o1, atol=1e-13, rtol=0)
    perm = np.array([(r % N) * P + r // N for r in range(P * N)])   # j-major row -> t-major row
    np.testing.assert_allclose(w1[:, :, perm][:, :, :, perm], w0, atol=1e-15, rtol=0)


@pytest.mark.parametrize("mask_mode,window", [(1, 0), (2, 2)])
def test_prefix_isolation(mask_mode, window):
    """"注意力机制" section 5.4 (prefix isolation): under a causal mask, changing
    inputs after position t0 leaves outputs at positions <= t0 unchanged."""
    rng = np.random.default_rng(700)
    B, N, H, d, P, t0 = 1, 8, 2, 3, 2, 4
    p = rand_problem(rng, B, N, H, d, P)
    a = run(oracle.get(), p, H, d, P, mask_mode=mask_mode, window=window)
    q = dict(p)
    q["X"] = p["X"].copy()
    q["X"][:, t0 + 1:] = rng.standard_normal(q["X"][:, t0 + 1:].shape) * 3
    b = run(oracle.get(), q, H, d, P, mask_mode=mask_mode, window=window)
    assert np.array_equal(a[:, :t0 + 1], b[:, :t0 + 1])
    assert not np.allclose(a[:, t0 + 1:], b[:, t0 + 1:])


def test_window_at_least_n_is_causal():
    rng = np.random.default_rng(800)
    B, N, H, d, P = 1, 6, 2, 3, 2
    p = rand_problem(rng, B, N, H, d, P)
    c = run(oracle.get(), p, H, d, P, mask_mode=1)
    for w in (N, N + 5):
        assert np.array_equal(run(oracle.get(), p, H, d, P, mask_mode=2, window=w), c)


def window_one_closed_form(p, H, d, P):
    """Window 1: pseudo-token (j, t) reads only the P pseudo-tokens of its own
    position t, so each row is a P-way softmax over j' at that t."""
    X = p["X"][0]
    N = X.shape[0]
    def mixed(W, alpha):
        base = np.stack([X @ W[:, m * d:(m + 1) * d] for m in range(H)])   # [m, t, c]
        return np.einsum("mhj,mtc->hjtc", alpha, base)
    q, k, v = mixed(p["W_Q"], p["alpha_Q"]), mixed(p["W_K"], p["alpha_K"]), mixed(p["W_V"], p["alpha_V"])
    out = np.zeros((N, H, d))
    for t in range(N):
        pbar = np.zeros((H, P, d))
        for h in range(H):
            for j in range(P):
                logits = np.array([q[h, j, t] @ k[h, j2, t] for j2 in range(P)]) / math.sqrt(d)
                w = np.exp(logits - logits.max())
                pbar[h, j] = (w / w.sum()) @ v[h, :, t]
        for h in range(H):
            for h2 in range(H):
                for j in range(P):
                    out[t, h] += p["R"][h, h2 * P + j] * pbar[h2, j]
    return out.reshape(1, N, H * d)


def check_window_one(orc, projection="c"):
    """The window's edge: t - t' < w with w = 1 admits t' = t only."""
    rng = np.random.default_rng(900)
    B, N, H, d, P = 1, 5, 2, 3, 3
    p = rand_problem(rng, B, N, H, d, P)
    got = run(orc, p, H, d, P, mask_mode=2, window=1, projection=projection)
    np.testing.assert_allclose(got, window_one_closed_form(p, H, d, P), atol=1e-12, rtol=0)


@pytest.mark.parametrize("projection", ["c", "numpy"])
def test_window_one_closed_form(projection):
    check_window_one(oracle.get(), projection)


def test_linear_in_R_and_alpha_V():
    """Step 4 is linear in R; steps 1-3 are linear in alpha_V (values enter the
    softmax read linearly)."""
    rng = np.random.default_rng(1000)
    B, N, H, d, P = 1, 5, 2, 3, 2
    p = rand_problem(rng, B, N, H, d, P)
    R2 = rng.standard_normal(p["R"].shape)
    f = lambda **kw: run(oracle.get(), dict(p, **kw), H, d, P, mask_mode=1)
    np.testing.assert_allclose(f(R=p["R"] + 2 * R2), f() + 2 * f(R=R2), atol=1e-12)
    A2 = rng.standard_normal(p["alpha_V"].shape)
    np.testing.assert_allclose(f(alpha_V=p["alpha_V"] - 3 * A2), f() - 3 * f(alpha_V=A2), atol=1e-12)


def test_projection_modes_agree():
    """The C projection loop and the library-matmul projection give the same
    forward pass (rounding only)."""
    rng = np.random.default_rng(1050)
    B, N, H, d, P = 2, 11, 3, 4, 2
    p = rand_problem(rng, B, N, H, d, P)
    for mm, w in MASKS:
        a = run(oracle.get(), p, H, d, P, mask_mode=mm, window=w, projection="c")
        b = run(oracle.get(), p, H, d, P, mask_mode=mm, window=w, projection="numpy")
        np.testing.assert_allclose(a, b, atol=1e-13, rtol=0)


def test_selected_rows_match_full_run():
    """Computing a subset of output rows gives the same values as the full run."""
    rng = np.random.default_rng(1100)
    B, N, H, d, P = 2, 9, 2, 3, 2
    p = rand_problem(rng, B, N, H, d, P)
    for mm, w in MASKS:
        full = run(oracle.get(), p, H, d, P, mask_mode=mm, window=w)
        rows = [0, 3, 8, 9, 13, 17]
        part = run(oracle.get(), p, H, d, P, mask_mode=mm, window=w, rows=rows)
        np.testing.assert_allclose(part, full.reshape(B * N, -1)[rows], atol=1e-14, rtol=0)


def test_brute_force_dense_matrices():
    """Algorithm 1 written once more as whole-matrix algebra on a tiny problem:
    mix, stack j-major, add a {0, -inf} mask on t, row softmax, unstack, contract."""
    rng = np.random.default_rng(1200)
    B, N, H, d, P = 1, 5, 2, 3, 2
    p = rand_problem(rng, B, N, H, d, P)
    X = p["X"][0]
    for mm, w in MASKS:
        def stacked(W, alpha):
            heads = [X @ W[:, m * d:(m + 1) * d] for m in range(H)]
            return [np.concatenate([sum(alpha[m, h, j] * heads[m] for m in range(H)) for j in range(P)])
                    for h in range(H)]
        Qb, Kb, Vb = stacked(p["W_Q"], p["alpha_Q"]), stacked(p["W_K"], p["alpha_K"]), stacked(p["W_V"], p["alpha_V"])
        tpos = np.tile(np.arange(N), P)
        M = np.zeros((P * N, P * N))
        if mm >= 1:
            M[tpos[None, :] > tpos[:, None]] = -np.inf
        if mm == 2:
            M[(tpos[:, None] - tpos[None, :]) >= w] = -np.inf
        Pb = []
        for h in range(H):
            S = Qb[h] @ Kb[h].T / math.sqrt(d) + M
            A = np.exp(S - S.max(axis=1, keepdims=True))
            A /= A.sum(axis=1, keepdims=True)
            Pb.append(A @ Vb[h])
        O = np.zeros((N, H, d))
        for h in range(H):
            for h2 in range(H):
                for j in range(P):
                    O[:, h] += p["R"][h, h2 * P + j] * Pb[h2][j * N:(j + 1) * N]
        got = run(oracle.get(), p, H, d, P, mask_mode=mm, window=w)
        np.testing.assert_allclose(got[0], O.reshape(N, H * d), atol=1e-12, rtol=0)


# ---------------------------------------------------------------------------
# The pins above catch planted mistakes
# ---------------------------------------------------------------------------

MUTANTS = {
    "scale by sqrt(D) instead of sqrt(d)":
        ("const double scale = 1.0 / sqrt((double)d);", "const double scale = 1.0 / sqrt((double)(c->H * d));"),
    "no softmax normalisation":
        ("double aj = allowed[j] ? exp(u[j] - c) / z : 0.0;", "double aj = allowed[j] ? exp(u[j] - c) : 0.0;"),
    "R indexed j*H + h'":
        ("const double rr = c->R[(i64)h * (H * P) + h2 * P + j];", "const double rr = c->R[(i64)h * (H * P) + j * H + h2];"),
    "alpha indexed [h][m][j]":
        ("const double a = c->alpha[s][((i64)m * H + h) * P + j];", "const double a = c->alpha[s][((i64)h * H + m) * P + j];"),
    "window admits t - t' == w":
        ("if (mask_mode == 2 && tq - tk >= window) return 0;", "if (mask_mode == 2 && tq - tk > window) return 0;"),
    "causal mask on the stacked row index":
        ("al[n] = (unsigned char)visible(c->mask_mode, c->window, t, c->klo + s2);",
         "al[n] = (unsigned char)(c->mask_mode == 0 || n <= j * nt + (t - c->klo));"),
    "keys mixed with alpha_Q":
        ("const double a = c->alpha[s][((i64)m * H + h) * P + j];",
         "const double a = c->alpha[s == 1 ? 0 : s][((i64)m * H + h) * P + j];"),
    "values taken from the keys":
        ("const double *Vh = c->mixed[2] + (i64)h * P * nt * d;", "const double *Vh = c->mixed[1] + (i64)h * P * nt * d;"),
    "contraction drops pseudo-blocks j > 0":
        ("            for (int j = 0; j < P; j++) {\n                const double rr",
         "            for (int j = 0; j < 1; j++) {\n                const double rr"),
}


def _pin_suite(orc, g):
    checks = [lambda: check_worked_example_causal(orc, g),
              lambda: check_scale_is_head_dim(orc, g),
              lambda: check_window_one(orc),
              lambda: check_window_one(orc, "numpy")]
    for P in (1, 2, 3):
        for mm, w in MASKS:
            checks.append(lambda P=P, mm=mm, w=w: check_contains_mha(orc, mm, w, P))
            checks.append(lambda P=P, mm=mm, w=w: check_repeated_tokens(orc, mm, w, P))
    failed = 0
    for c in checks:
        try:
            c()
        except (AssertionError, RuntimeError):
            failed += 1
    return failed


def test_planted_mistakes_are_caught(golden, tmp_path):
    """Each planted slip, compiled into a copy of the oracle, fails some pin
    (and the unmodified oracle fails none)."""
    g = golden("causal_single_head_example.txt")
    src = open(os.path.join(os.path.dirname(oracle.__file__), "iha_oracle.c")).read()
    assert _pin_suite(oracle.get(), g) == 0
    for i, (name, (old, new)) in enumerate(MUTANTS.items()):
        assert src.count(old) >= 1, f"mutation site missing: {name}"
        path = tmp_path / f"mutant{i}.c"
        path.write_text(src.replace(old, new, 1))
        lib = oracle.build(force=True, src=str(path), out=str(tmp_path / f"mutant{i}.so"))
        assert _pin_suite(oracle.Oracle(lib), g) > 0, f"planted mistake not caught: {name}"


# ---------------------------------------------------------------------------
# the backward oracle (oracle/backward.py): its forward is the pinned C oracle's, and its
# gradients are the derivatives of that forward (central finite differences)
# ---------------------------------------------------------------------------

BWD_CASES = [
    # B, N, H, d, P, mask_mode, window
    (2, 9, 3, 4, 2, 1, 0),
    (1, 7, 2, 5, 3, 2, 3),
    (1, 6, 2, 4, 1, 0, 0),
    (2, 5, 2, 3, 4, 2, 1),
]


@pytest.mark.parametrize("case", BWD_CASES)
def test_backward_oracle_forward_is_the_c_oracle(case):
    """The autograd graph is Algorithm 1 as the C oracle computes it (same inputs, float64)."""
    import torch
    from oracle import backward as bwd
    B, N, H, d, P, mode, w = case
    p = rand_problem(RNG, B, N, H, d, P)
    ref = run(oracle, p, H, d, P, mask_mode=mode, window=w)
    got = bwd.forward(*(torch.as_tensor(p[k]) for k in bwd.PARAMS), H=H, d=d, P=P, mask_mode=mode,
                      window=w).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("case", BWD_CASES)
def test_backward_oracle_matches_finite_differences(case):
    """<grad, v> equals the central difference of <out, dO> along a random direction v, for
    every input of Algorithm 1 (X, the three W, the three alpha, R)."""
    import torch
    from oracle import backward as bwd
    B, N, H, d, P, mode, w = case
    rng = np.random.default_rng(777 + P)
    p = rand_problem(rng, B, N, H, d, P)
    dO = rng.standard_normal((B, N, H * d))
    grads = bwd.backward(p, dO, H=H, d=d, P=P, mask_mode=mode, window=w)

    def f(q):
        out = bwd.forward(*(torch.as_tensor(q[k]) for k in bwd.PARAMS), H=H, d=d, P=P, mask_mode=mode, window=w)
        return float((out.numpy() * dO).sum())

    eps = 1e-6
    for k in bwd.PARAMS:
        v = rng.standard_normal(np.shape(p[k]))
        plus = dict(p, **{k: p[k] + eps * v})
        minus = dict(p, **{k: p[k] - eps * v})
        fd = (f(plus) - f(minus)) / (2 * eps)
        an = float((grads[k].numpy() * v).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (k, fd, an)


def test_cancellation_scale_closed_form():
    """One token, one head, P = 1: the softmax has one entry (p = 1), so the term P*D alone
    is -D with D = dPbar . v, v = alpha_V x W_V, dPbar = R dO; through s = (alpha_Q x W_Q) .
    (alpha_K x W_K) / sqrt(d) it gives dW_Q[i][c] = -D alpha_Q alpha_K x_i (x W_K)_c / sqrt(d)
    and symmetrically for W_K, X and the alphas; the value-path inputs get nothing."""
    import torch
    from oracle import backward as bwd
    rng = np.random.default_rng(5)
    d = 6
    p = rand_problem(rng, 1, 1, 1, d, 1)
    dO = rng.standard_normal((1, 1, d))
    sc = bwd.cancellation_scale(p, dO, H=1, d=d, P=1, mask_mode=1)
    x = p["X"][0, 0]
    aq, ak, av, r = p["alpha_Q"][0, 0, 0], p["alpha_K"][0, 0, 0], p["alpha_V"][0, 0, 0], p["R"][0, 0]
    yq, yk, yv = x @ p["W_Q"], x @ p["W_K"], x @ p["W_V"]
    D = float((r * dO[0, 0]) @ (av * yv))
    g = -D / np.sqrt(d)
    np.testing.assert_allclose(sc["W_Q"].numpy(), g * aq * ak * np.outer(x, yk), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(sc["W_K"].numpy(), g * aq * ak * np.outer(x, yq), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(sc["X"].numpy()[0, 0], g * aq * ak * (p["W_Q"] @ yk + p["W_K"] @ yq), rtol=1e-10,
                               atol=1e-12)
    np.testing.assert_allclose(float(sc["alpha_Q"].numpy()[0, 0, 0]), g * ak * float(yq @ yk), rtol=1e-10)
    np.testing.assert_allclose(float(sc["alpha_K"].numpy()[0, 0, 0]), g * aq * float(yq @ yk), rtol=1e-10)
    for k in ("W_V", "alpha_V", "R"):
        assert not sc[k].numpy().any(), k


@pytest.mark.parametrize("case", BWD_CASES)
def test_cancellation_scale_linear_in_dO(case):
    """The scale is linear in dO (D is) and zero for the value-path inputs at any shape."""
    from oracle import backward as bwd
    B, N, H, d, P, mode, w = case
    rng = np.random.default_rng(888 + P)
    p = rand_problem(rng, B, N, H, d, P)
    d1, d2 = rng.standard_normal((2, B, N, H * d))
    s1 = bwd.cancellation_scale(p, d1, H=H, d=d, P=P, mask_mode=mode, window=w)
    s2 = bwd.cancellation_scale(p, d2, H=H, d=d, P=P, mask_mode=mode, window=w)
    s12 = bwd.cancellation_scale(p, 2.0 * d1 - d2, H=H, d=d, P=P, mask_mode=mode, window=w)
    for k in bwd.PARAMS:
        np.testing.assert_allclose(s12[k].numpy(), 2.0 * s1[k].numpy() - s2[k].numpy(), rtol=1e-9,
                                   atol=1e-9 * (1 + np.abs(s1[k].numpy()).max()))
    for k in ("W_V", "alpha_V", "R"):
        assert not s1[k].numpy().any(), k


def test_gram_term_scale_closed_form_and_bounds():
    """gram_term_scale, the tolerance scale of the four token-sum gradients:
    - one token, one head, P = 1, d columns: dR = sum_c dO_c Pbar_c with Pbar = v (the one
      readable value, p = 1) = alpha_V x W_V, so its scale is sqrt(sum_c (dO_c v_c)^2); dalpha_V
      = sum_c (x W_V)_c dv_c with dv = R dO, scale sqrt(sum_c ((x W_V)_c R dO_c)^2);
    - at any shape each gradient is at most sqrt(number of terms) times its scale
      (Cauchy-Schwarz), the scale is linear in |dO| and, for dR, independent of R."""
    from oracle import backward as bwd
    rng = np.random.default_rng(17)
    d = 5
    p = rand_problem(rng, 1, 1, 1, d, 1)
    dO = rng.standard_normal((1, 1, d))
    sc = bwd.gram_term_scale(p, dO, H=1, d=d, P=1, mask_mode=1)
    x = p["X"][0, 0]
    yv = x @ p["W_V"]
    v = p["alpha_V"][0, 0, 0] * yv
    r = p["R"][0, 0]
    np.testing.assert_allclose(float(sc["R"].numpy()[0, 0]), np.sqrt(np.sum((dO[0, 0] * v) ** 2)), rtol=1e-12)
    np.testing.assert_allclose(float(sc["alpha_V"].numpy()[0, 0, 0]), np.sqrt(np.sum((yv * r * dO[0, 0]) ** 2)),
                               rtol=1e-12)
    for case in BWD_CASES[:3]:
        B, N, H, d, P, mode, w = case
        rng = np.random.default_rng(99 + N)
        p = rand_problem(rng, B, N, H, d, P)
        dO = rng.standard_normal((B, N, H * d))
        sc = bwd.gram_term_scale(p, dO, H=H, d=d, P=P, mask_mode=mode, window=w)
        ref = bwd.backward(p, dO, H=H, d=d, P=P, mask_mode=mode, window=w)
        n = B * N * d
        for k, s in sc.items():
            assert (np.abs(ref[k].numpy()) <= np.sqrt(n) * s.numpy() * (1 + 1e-9) + 1e-12).all(), k
        sc3 = bwd.gram_term_scale(p, -3.0 * dO, H=H, d=d, P=P, mask_mode=mode, window=w)
        for k in sc:
            np.testing.assert_allclose(sc3[k].numpy(), 3.0 * sc[k].numpy(), rtol=1e-10, atol=1e-300)
        p2 = dict(p)
        p2["R"] = 2.0 * p["R"]
        sc_r = bwd.gram_term_scale(p2, dO, H=H, d=d, P=P, mask_mode=mode, window=w)
        np.testing.assert_allclose(sc_r["R"].numpy(), sc["R"].numpy(), rtol=1e-10, atol=1e-300)
        np.testing.assert_allclose(sc_r["alpha_V"].numpy(), 2.0 * sc["alpha_V"].numpy(), rtol=1e-10, atol=1e-300)
