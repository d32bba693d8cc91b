"""Pins of the oracle's backward pass (fp64): central finite differences of
the loss sum(O * dO), torch autograd in fp64 on an independent softmax
attention, and the closed form sum_j dV_j = sum_i dO_i (rows of P sum to 1)."""
import numpy as np
import pytest
import torch

import oracle


def _inputs(B, Hq, Hkv, nq, nkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s: torch.randn(*s, generator=g, dtype=torch.float64)  # noqa: E731
    return mk(B, Hq, nq, d), mk(B, Hkv, nkv, d), mk(B, Hkv, nkv, d), mk(B, Hq, nq, d)


def _loss(Q, K, V, dO, causal):
    O, _ = oracle.sdpa(Q, K, V, causal)
    return float((O * dO.numpy()).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_central_differences(causal):
    Q, K, V, dO = _inputs(1, 4, 2, 6, 9, 5, seed=1)
    dQ, dK, dV = oracle.backward(Q, K, V, dO, causal)
    rng = np.random.default_rng(0)
    eps = 1e-5
    for X, G in ((Q, dQ), (K, dK), (V, dV)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in X.shape)
            Xp, Xm = X.clone(), X.clone()
            Xp[idx] += eps
            Xm[idx] -= eps
            args_p = [Xp if Y is X else Y for Y in (Q, K, V)]
            args_m = [Xm if Y is X else Y for Y in (Q, K, V)]
            fd = (_loss(*args_p, dO, causal) - _loss(*args_m, dO, causal)) / (2 * eps)
            assert abs(fd - G[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, G[idx])


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd(causal):
    B, Hq, Hkv, nq, nkv, d = 2, 4, 2, 7, 11, 8
    Q, K, V, dO = _inputs(B, Hq, Hkv, nq, nkv, d, seed=2)
    G = Hq // Hkv
    q, k, v = (x.clone().requires_grad_(True) for x in (Q, K, V))
    kk, vv = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    s = (q @ kk.transpose(-1, -2)) / np.sqrt(d)
    if causal:
        i = torch.arange(nq)[:, None]
        j = torch.arange(nkv)[None, :]
        s = s.masked_fill(j > i + (nkv - nq), float("-inf"))
    (torch.softmax(s, dim=-1) @ vv).backward(dO)
    dQ, dK, dV = oracle.backward(Q, K, V, dO, causal)
    assert np.allclose(dQ, q.grad.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(dK, k.grad.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(dV, v.grad.numpy(), rtol=0, atol=1e-12)


def test_backward_dv_column_sums_and_magnitudes():
    Q, K, V, dO = _inputs(1, 2, 1, 10, 10, 4, seed=3)
    dQ, dK, dV, (mq, mk, mv) = oracle.backward(Q, K, V, dO, False, magnitudes=True)
    # sum over keys of dV = sum over the rows (and the G heads) of dO
    assert np.allclose(dV.sum(axis=2), dO.numpy().sum(axis=2).sum(axis=1, keepdims=True),
                       atol=1e-12)
    # each gradient is bounded by the sum of the magnitudes of its terms
    assert (np.abs(dQ) <= mq + 1e-15).all() and (np.abs(dK) <= mk + 1e-15).all()
    assert (np.abs(dV) <= mv + 1e-15).all()


def test_backward_d_sensitivity_bounds_a_perturbed_d():
    """dsens_q / dsens_k bound the change of dQ / dK when every D_i moves by
    up to d_err_i: perturb D directly (dS = P (dP - D - delta)) and compare."""
    B, Hq, Hkv, nq, nkv, d = 1, 2, 1, 5, 7, 4
    Q, K, V, dO = _inputs(B, Hq, Hkv, nq, nkv, d, seed=4)
    scale = 1.0 / np.sqrt(d)
    rng = np.random.default_rng(1)
    delta = rng.uniform(-1, 1, (B, Hq, nq)) * 0.01
    dQ, dK, _, (_, _, _, sq, sk) = oracle.backward(Q, K, V, dO, True, magnitudes=True,
                                                   d_err=np.abs(delta))
    # reference: the same gradients with D_i replaced by D_i + delta_i
    G = Hq // Hkv
    kk = K.repeat_interleave(G, dim=1).numpy()
    vv = V.repeat_interleave(G, dim=1).numpy()
    q, go = Q.numpy(), dO.numpy()
    s = q @ kk.transpose(0, 1, 3, 2) * scale
    i, j = np.arange(nq)[:, None], np.arange(nkv)[None, :]
    s = np.where(j > i + (nkv - nq), -np.inf, s)
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    dp = go @ vv.transpose(0, 1, 3, 2)
    D = (p * dp).sum(-1, keepdims=True) + delta[..., None]
    ds = p * (dp - D)
    dQ2 = scale * ds @ kk
    dK2 = (scale * ds.transpose(0, 1, 3, 2) @ q).reshape(B, Hkv, G, nkv, d).sum(2)
    assert (np.abs(dQ2 - dQ) <= sq + 1e-12).all()
    assert (np.abs(dK2 - dK) <= sk + 1e-12).all()
    assert np.abs(dQ2 - dQ).max() > 0.1 * sq.max()   # the bound is not vacuous
