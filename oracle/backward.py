"""fp64 CPU oracle of the Interleaved Head Attention backward pass.

TEST INFRASTRUCTURE ONLY: the tests and the benchmark's CPU leg call it; the product never
does.  It shares no code with the CUDA path.

Algorithm 1 ("Interleaved Head Attention" section 4) is written again here in plain PyTorch
float64 CPU operations, step by step: the per-head projections X W_s^(m), the pseudo-head
mixing with alpha_s, the j-major stacking of the P pseudo-blocks into a sequence of length
P*N, masked softmax attention per head over that sequence (dense, the operator of
"注意力机制" eq. (5.11); the mask reads the original position t of each stacked row),
unstacking, and the R contraction with the heads concatenated.  The gradients of the output
with respect to X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V and R are torch.autograd's chain
rule through exactly these steps (for the softmax part the derivatives of
"注意力机制" eqs. (5.24)-(5.31)).

Pinned by tests/test_oracle_pins.py: its forward equals the C oracle's (itself pinned to
the pages), and its gradients equal central finite differences of that forward.
"""
from __future__ import annotations

import math

import torch

PARAMS = ("X", "W_Q", "W_K", "W_V", "alpha_Q", "alpha_K", "alpha_V", "R")


def _allowed(N: int, P: int, mask_mode: int, window: int) -> torch.Tensor:
    """allowed[r, c] for j-major stacked rows r = j*N + t (original position t = r % N)."""
    t = torch.arange(P * N) % N
    tq, tk = t[:, None], t[None, :]
    ok = torch.ones(P * N, P * N, dtype=torch.bool)
    if mask_mode >= 1:
        ok &= tk <= tq
    if mask_mode == 2:
        ok &= (tq - tk) < window
    return ok


def forward(X, W_Q, W_K, W_V, alpha_Q, alpha_K, alpha_V, R, *, H, d, P, mask_mode=0, window=0):
    """out [B, N, H*d] of Algorithm 1 in float64 torch ops (differentiable)."""
    B, N, D = X.shape
    ok = _allowed(N, P, mask_mode, window)

    def pseudo(W, alpha):
        Y = (X @ W).reshape(B, N, H, d)                          # X W^(m): [b, t, m, c]
        S = torch.einsum("mhj,btmc->bhjtc", alpha, Y)             # sum_m alpha[m,h,j] X W^(m)
        return S.reshape(B, H, P * N, d)                          # j-major stacking: row j*N + t

    Qb, Kb, Vb = pseudo(W_Q, alpha_Q), pseudo(W_K, alpha_K), pseudo(W_V, alpha_V)
    S = (Qb @ Kb.transpose(-1, -2)) / math.sqrt(d)
    S = S.masked_fill(~ok, float("-inf"))
    A = torch.softmax(S, dim=-1)
    Pb = A @ Vb                                                   # [b, h', j*N + t, c]
    Pu = Pb.reshape(B, H, P, N, d).reshape(B, H * P, N, d)        # unstack: index h'*P + j
    O = torch.einsum("hk,bktc->bthc", R, Pu)                      # sum R[h, h'P+j] P_{h',j}[t]
    return O.reshape(B, N, H * d)


def cancellation_scale(inputs: dict, dO, *, H, d, P, mask_mode=0, window=0):
    """The gradients of every input reached through the scores by the term P * D alone, where
    D_r = dPbar_r . Pbar_r: the softmax derivative ("注意力机制" eqs. (5.24)-(5.31)) gives
    dS = P * (dP - D), and D computed from a rounded attention output carries a relative
    error that dS inherits at the size of P * D, not of dS (which may cancel to 0).  These
    tensors set the absolute scale of that error in a tolerance; float64, keys of PARAMS
    (zeros for the inputs the scores do not depend on)."""
    leaves = {k: torch.as_tensor(inputs[k], dtype=torch.float64).clone().requires_grad_(True) for k in PARAMS}
    X, W_Q, W_K, W_V = leaves["X"], leaves["W_Q"], leaves["W_K"], leaves["W_V"]
    B, N, D_ = X.shape
    ok = _allowed(N, P, mask_mode, window)

    def pseudo(W, alpha):
        Y = (X @ W).reshape(B, N, H, d)
        return torch.einsum("mhj,btmc->bhjtc", alpha, Y).reshape(B, H, P * N, d)

    Qb, Kb = pseudo(W_Q, leaves["alpha_Q"]), pseudo(W_K, leaves["alpha_K"])
    Vb = pseudo(W_V, leaves["alpha_V"]).detach()
    S = ((Qb @ Kb.transpose(-1, -2)) / math.sqrt(d)).masked_fill(~ok, float("-inf"))
    A = torch.softmax(S, dim=-1).detach()
    Pb = (A @ Vb).requires_grad_(True)
    Pu = Pb.reshape(B, H, P, N, d).reshape(B, H * P, N, d)
    O = torch.einsum("hk,bktc->bthc", leaves["R"].detach(), Pu).reshape(B, N, H * d)
    (dPb,) = torch.autograd.grad(O, Pb, torch.as_tensor(dO, dtype=torch.float64))
    Dr = (dPb * Pb.detach()).sum(-1, keepdim=True)
    S_fin = S.masked_fill(~ok, 0.0)   # the masked entries carry no gradient (A = 0 there)
    grads = torch.autograd.grad(S_fin, [leaves[k] for k in PARAMS], -(A * Dr), allow_unused=True)
    return {k: (g.detach() if g is not None else torch.zeros_like(leaves[k])) for k, g in zip(PARAMS, grads)}


def backward(inputs: dict, dO, *, H, d, P, mask_mode=0, window=0):
    """Gradients of sum(out * dO) for every input of Algorithm 1; float64 numpy-compatible
    tensors in, a dict of float64 tensors (same keys as PARAMS) out."""
    leaves = {k: torch.as_tensor(inputs[k], dtype=torch.float64).clone().requires_grad_(True) for k in PARAMS}
    out = forward(*(leaves[k] for k in PARAMS), H=H, d=d, P=P, mask_mode=mask_mode, window=window)
    grads = torch.autograd.grad(out, [leaves[k] for k in PARAMS], torch.as_tensor(dO, dtype=torch.float64))
    return {k: g.detach() for k, g in zip(PARAMS, grads)}


def gram_term_scale(inputs: dict, dO, *, H, d, P, mask_mode=0, window=0):
    """The size of the individual terms of the four gradients that are sums over every token
    and column of a product of two stored tensors (chain rule through Algorithm 1's mixing and
    contraction steps):
        dalpha_s[m,h,j] = sum_{t,c} (X W_s^(m))[t,c] * dS~_s[h,j][t,c]
        dR[h, h'P+j]    = sum_{t,c} dO_h[t,c] * P_{h',j}[t,c]
    For each output element, sqrt(sum over (t,c) of term^2): the standard deviation of the sum's
    error when each term carries an independent relative error of 1 (the factors are stored in
    bfloat16).  Where the terms cancel, the result can be far smaller than this scale, and a
    tolerance relative to the result alone is ill-conditioned.  float64; keys alpha_Q, alpha_K,
    alpha_V, R (the other keys are not such sums and are absent)."""
    f = {k: torch.as_tensor(inputs[k], dtype=torch.float64) for k in PARAMS}
    X = f["X"]
    B, N, D_ = X.shape
    ok = _allowed(N, P, mask_mode, window)
    Y = {s: (X @ f["W_" + s]).reshape(B, N, H, d) for s in ("Q", "K", "V")}
    mixed = {s: torch.einsum("mhj,btmc->bhjtc", f["alpha_" + s], Y[s]).reshape(B, H, P * N, d).requires_grad_(True)
             for s in ("Q", "K", "V")}
    S = (mixed["Q"] @ mixed["K"].transpose(-1, -2)) / math.sqrt(d)
    A = torch.softmax(S.masked_fill(~ok, float("-inf")), dim=-1)
    Pb = A @ mixed["V"]
    Pu = Pb.reshape(B, H, P, N, d).reshape(B, H * P, N, d)
    O = torch.einsum("hk,bktc->bthc", f["R"], Pu).reshape(B, N, H * d)
    dOt = torch.as_tensor(dO, dtype=torch.float64)
    g = torch.autograd.grad(O, [mixed[s] for s in ("Q", "K", "V")], dOt)
    out = {}
    for s, gs in zip(("Q", "K", "V"), g):
        dS = gs.detach().reshape(B, H, P, N, d)                    # [b, h, j, t, c]
        out["alpha_" + s] = torch.einsum("btmc,bhjtc->mhj", Y[s] ** 2, dS ** 2).sqrt()
    Pd = Pu.detach().reshape(B, H * P, N, d)
    out["R"] = torch.einsum("bthc,bktc->hk", dOt.reshape(B, N, H, d) ** 2, Pd ** 2).sqrt()
    return out
