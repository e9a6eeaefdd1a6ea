"""Pins for the fp64 oracle: each check fixes the oracle to something other
than itself (finite differences, exact symbolic differentiation, a library
routine, a closed form, an exact invariant or a loop-only brute force)."""
import numpy as np
import pytest

from oracle import bob as orc

RTOL_FD = 2e-7


def rand_inputs(N, d, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return [scale * rng.standard_normal((N, d)) for _ in range(7)]


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# --------------------------------------------------------------------------
# forward / prep / first backward
# --------------------------------------------------------------------------

def test_forward_matches_scipy_softmax():
    from scipy.special import logsumexp, softmax
    Q, K, V, *_ = rand_inputs(9, 4, 1)
    tau = 0.37
    S, P, O, L = orc.forward(Q, K, V, tau)
    assert np.allclose(S, tau * np.einsum("ik,jk->ij", Q, K), rtol=1e-14, atol=1e-14)
    assert np.allclose(L, logsumexp(S, axis=1), rtol=1e-14)
    assert np.allclose(P, softmax(S, axis=1), rtol=1e-13)
    assert np.allclose(P.sum(axis=1), 1.0, atol=1e-14)
    assert np.allclose(O, np.einsum("ij,jk->ik", softmax(S, axis=1), V), rtol=1e-13)


def test_prep_D_is_rowsum_P_dP():
    Q, K, V, dO, *_ = rand_inputs(11, 5, 2)
    tau = 0.5
    O, L, D = orc.prep(Q, K, V, dO, tau)
    _, P, _, _ = orc.forward(Q, K, V, tau)
    dP = dO @ V.T
    assert np.allclose(D, (P * dP).sum(axis=1), rtol=1e-12, atol=1e-13)


def _fd_grad(fun, X, h=1e-5):
    g = np.zeros_like(X)
    for idx in np.ndindex(*X.shape):
        Xp = X.copy()
        Xm = X.copy()
        Xp[idx] += h
        Xm[idx] -= h
        g[idx] = (fun(Xp) - fun(Xm)) / (2 * h)
    return g


def test_first_backward_matches_fd_of_output_inner_product():
    Q, K, V, dO, *_ = rand_inputs(6, 3, 3)
    tau = 0.6
    dQ, dK, dV = orc.first_backward(Q, K, V, dO, tau)

    def psi(Q_, K_, V_):
        return float((orc.forward(Q_, K_, V_, tau)[2] * dO).sum())

    assert rel(dQ, _fd_grad(lambda X: psi(X, K, V), Q)) < RTOL_FD
    assert rel(dK, _fd_grad(lambda X: psi(Q, X, V), K)) < RTOL_FD
    assert rel(dV, _fd_grad(lambda X: psi(Q, K, X), V)) < RTOL_FD


def test_first_backward_matches_torch_autograd():
    torch = pytest.importorskip("torch")
    Q, K, V, dO, *_ = rand_inputs(13, 6, 4)
    tau = 1 / np.sqrt(6)
    dQ, dK, dV = orc.first_backward(Q, K, V, dO, tau)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
    out = torch.softmax(tau * tq @ tk.T, dim=-1) @ tv
    gq, gk, gv = torch.autograd.grad(out, (tq, tk, tv), torch.tensor(dO))
    assert rel(dQ, gq.numpy()) < 1e-13
    assert rel(dK, gk.numpy()) < 1e-13
    assert rel(dV, gv.numpy()) < 1e-13


# --------------------------------------------------------------------------
# BoB against finite differences of Phi
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,d,seed,tau", [(7, 5, 0, 1 / np.sqrt(5)), (16, 8, 1, 0.35),
                                          (3, 2, 2, 1.3), (12, 4, 3, 0.5)])
def test_bob_matches_fd_of_phi(N, d, seed, tau):
    Q, K, V, dO, UQ, UK, UV = rand_inputs(N, d, seed)
    r = orc.bob(Q, K, V, dO, UQ, UK, UV, tau)
    args = [Q, K, V, dO]
    for pos, key in enumerate(("dQt", "dKt", "dVt", "ddOt")):
        def f(X, pos=pos):
            a = list(args)
            a[pos] = X
            return orc.phi(*a, UQ, UK, UV, tau)
        assert rel(r[key], _fd_grad(f, args[pos])) < RTOL_FD, key


def test_bob_matches_fd_with_peaked_rows():
    # large scores: nearly one-hot softmax rows
    Q, K, V, dO, UQ, UK, UV = rand_inputs(8, 3, 5)
    Q = 3.0 * Q
    K[2] *= 4.0
    tau = 1.0
    r = orc.bob(Q, K, V, dO, UQ, UK, UV, tau)
    for pos, key in ((0, "dQt"), (1, "dKt")):
        args = [Q, K, V, dO]

        def f(X, pos=pos):
            a = list(args)
            a[pos] = X
            return orc.phi(*a, UQ, UK, UV, tau)
        assert rel(r[key], _fd_grad(f, args[pos], h=1e-6)) < 1e-6, key


# --------------------------------------------------------------------------
# Exact symbolic differentiation (sympy) on a tiny case
# --------------------------------------------------------------------------

def test_bob_matches_sympy_exact_derivative():
    sp = pytest.importorskip("sympy")
    N, d = 3, 2
    rng = np.random.default_rng(7)
    vals = [np.round(rng.standard_normal((N, d)), 3) for _ in range(7)]
    tau = sp.Rational(7, 10)

    def mat(name):
        return sp.Matrix(N, d, lambda i, k: sp.Symbol(f"{name}_{i}_{k}"))

    Qs, Ks, Vs, dOs = mat("Q"), mat("K"), mat("V"), mat("dO")
    UQ, UK, UV = (sp.Matrix(v.tolist()).applyfunc(sp.nsimplify) for v in vals[4:])
    S = tau * Qs * Ks.T
    Pm = sp.Matrix(N, N, lambda i, j: sp.exp(S[i, j]) / sum(sp.exp(S[i, c]) for c in range(N)))
    Om = Pm * Vs
    dV = Pm.T * dOs
    dP = dOs * Vs.T
    Dv = [sum(Pm[i, j] * dP[i, j] for j in range(N)) for i in range(N)]
    dS = sp.Matrix(N, N, lambda i, j: Pm[i, j] * (dP[i, j] - Dv[i]))
    dQ = tau * dS * Ks
    dK = tau * dS.T * Qs
    Phi = sum(dQ[i, k] * UQ[i, k] + dK[i, k] * UK[i, k] + dV[i, k] * UV[i, k]
              for i in range(N) for k in range(d))
    subs = {}
    for M, v in zip((Qs, Ks, Vs, dOs), vals[:4]):
        for i in range(N):
            for k in range(d):
                subs[M[i, k]] = sp.nsimplify(v[i, k])
    r = orc.bob(*vals, float(tau))
    for M, key in ((Qs, "dQt"), (Ks, "dKt"), (Vs, "dVt"), (dOs, "ddOt")):
        exact = np.array([[float(sp.diff(Phi, M[i, k]).evalf(30, subs=subs))
                           for k in range(d)] for i in range(N)])
        assert rel(r[key], exact) < 1e-12, key
    del Om


# --------------------------------------------------------------------------
# Brute force, affine form, per-row form
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,d,seed", [(1, 3, 0), (5, 3, 1), (12, 6, 2)])
def test_bob_matches_bruteforce(N, d, seed):
    args = rand_inputs(N, d, seed)
    tau = 0.41
    r = orc.bob(*args, tau)
    b = orc.bob_bruteforce(*args, tau)
    for key in ("dQt", "dKt", "dVt", "ddOt", "alpha", "E"):
        assert rel(r[key], b[key]) < 1e-12, key


def test_affine_identities_of_the_row_outputs():
    # E = E0 - alpha D, d~dO = d~dO0 - alpha O, d~Q = tau (Omega - alpha R - E B)
    args = rand_inputs(40, 8, 11)
    tau = 1 / np.sqrt(8)
    r = orc.bob(*args, tau)
    a = orc.bob_affine(*args, tau)
    for key in ("dQt", "ddOt", "alpha", "E"):
        assert rel(a[key], r[key]) < 1e-12, key


def test_rows_form_matches_matrix_form():
    args = rand_inputs(37, 6, 12)
    tau = 0.4
    r = orc.bob(*args, tau)
    rows = [0, 5, 17, 36]
    s = orc.bob_rows(*args, tau, rows)
    for key in ("dQt", "ddOt", "alpha", "E", "L", "D"):
        assert rel(s[key], r[key][rows]) < 1e-12, key


# --------------------------------------------------------------------------
# Exact invariants and closed forms
# --------------------------------------------------------------------------

def test_invariants():
    Q, K, V, dO, UQ, UK, UV = rand_inputs(33, 7, 13)
    tau = 0.45
    r = orc.bob(Q, K, V, dO, UQ, UK, UV, tau)
    dQ, dK, dV = orc.first_backward(Q, K, V, dO, tau)
    ph = orc.phi(Q, K, V, dO, UQ, UK, UV, tau)
    scale = np.abs(ph) + 1.0
    # Phi is invariant under K -> K + 1 c^T and V -> V + 1 c^T
    assert np.abs(r["dKt"].sum(axis=0)).max() < 1e-12 * np.abs(r["dKt"]).max() * 33
    assert np.abs(r["dVt"].sum(axis=0)).max() < 1e-12 * np.abs(r["dVt"]).max() * 33
    # Phi is linear in dO
    assert abs((r["ddOt"] * dO).sum() - ph) < 1e-12 * scale
    # dQ and dK are linear in V and dV does not depend on V
    assert abs((r["dVt"] * V).sum() - ((dQ * UQ).sum() + (dK * UK).sum())) < 1e-12 * scale
    # Q -> sQ, K -> K/s leaves S unchanged
    lhs = (r["dQt"] * Q).sum() - (r["dKt"] * K).sum()
    rhs = (dK * UK).sum() - (dQ * UQ).sum()
    assert abs(lhs - rhs) < 1e-12 * scale


def test_linear_in_perturbations_and_zero_at_zero():
    Q, K, V, dO, UQ, UK, UV = rand_inputs(10, 4, 14)
    tau = 0.7
    W = rand_inputs(10, 4, 15)
    r1 = orc.bob(Q, K, V, dO, UQ, UK, UV, tau)
    r2 = orc.bob(Q, K, V, dO, W[0], W[1], W[2], tau)
    r12 = orc.bob(Q, K, V, dO, UQ + 2 * W[0], UK + 2 * W[1], UV + 2 * W[2], tau)
    for key in ("dQt", "dKt", "dVt", "ddOt", "alpha", "E"):
        assert rel(r12[key], r1[key] + 2 * r2[key]) < 1e-12, key
    z = np.zeros_like(Q)
    r0 = orc.bob(Q, K, V, dO, z, z, z, tau)
    for key in ("dQt", "dKt", "dVt", "ddOt", "alpha", "E"):
        assert np.abs(r0[key]).max() == 0.0, key


def test_hessian_symmetry():
    # (d~Q, d~K, d~V) = Hessian of psi = <Attn(Q,K,V), dO> applied to U
    Q, K, V, dO, UQ, UK, UV = rand_inputs(9, 3, 16)
    W = rand_inputs(9, 3, 17)[:3]
    tau = 0.8
    ru = orc.bob(Q, K, V, dO, UQ, UK, UV, tau)
    rw = orc.bob(Q, K, V, dO, *W, tau)
    a = sum((ru[k] * w).sum() for k, w in zip(("dQt", "dKt", "dVt"), W))
    b = sum((rw[k] * u).sum() for k, u in zip(("dQt", "dKt", "dVt"), (UQ, UK, UV)))
    assert abs(a - b) < 1e-12 * (abs(a) + 1)


def test_n_equals_one_closed_form():
    Q, K, V, dO, UQ, UK, UV = rand_inputs(1, 5, 18)
    tau = 0.3
    r = orc.bob(Q, K, V, dO, UQ, UK, UV, tau)
    alpha = tau * (UQ[0] @ K[0] + Q[0] @ UK[0])
    Dv = dO[0] @ V[0]
    # dS = 0 up to the rounding of dP - D (D is dO . O with O = V exactly)
    assert np.abs(r["dQt"]).max() < 1e-15 and np.abs(r["dKt"]).max() < 1e-15
    assert np.abs(r["dVt"]).max() < 1e-15
    assert np.allclose(r["ddOt"], UV, rtol=1e-14, atol=1e-15)
    assert np.isclose(r["alpha"][0], alpha, rtol=1e-14)
    assert np.isclose(r["E"][0], dO[0] @ UV[0] - alpha * Dv, rtol=1e-13, atol=1e-14)


def test_uq_uk_zero_reduces_to_first_backward_with_v_replaced():
    torch = pytest.importorskip("torch")
    Q, K, V, dO, _, _, UV = rand_inputs(14, 5, 19)
    tau = 1 / np.sqrt(5)
    z = np.zeros_like(Q)
    r = orc.bob(Q, K, V, dO, z, z, UV, tau)
    tq, tk, tu = (torch.tensor(x, requires_grad=True) for x in (Q, K, UV))
    att = torch.softmax(tau * tq @ tk.T, dim=-1) @ tu
    gq, gk = torch.autograd.grad(att, (tq, tk), torch.tensor(dO))
    assert rel(r["ddOt"], att.detach().numpy()) < 1e-13
    assert np.abs(r["dVt"]).max() == 0
    assert rel(r["dQt"], gq.numpy()) < 1e-12
    assert rel(r["dKt"], gk.numpy()) < 1e-12


def test_jvp_identities_of_the_forward():
    # d~dO is the JVP of O along (U_Q, U_K, U_V); alpha is the JVP of L
    Q, K, V, dO, UQ, UK, UV = rand_inputs(10, 4, 20)
    tau = 0.55
    r = orc.bob(Q, K, V, dO, UQ, UK, UV, tau)
    h = 1e-5
    _, _, Op, Lp = orc.forward(Q + h * UQ, K + h * UK, V + h * UV, tau)
    _, _, Om, Lm = orc.forward(Q - h * UQ, K - h * UK, V - h * UV, tau)
    assert rel(r["ddOt"], (Op - Om) / (2 * h)) < 1e-8
    assert rel(r["alpha"], (Lp - Lm) / (2 * h)) < 1e-8


def test_matches_torch_double_backward():
    torch = pytest.importorskip("torch")
    N, d = 24, 8
    args = rand_inputs(N, d, 21)
    tau = 1 / np.sqrt(d)
    r = orc.bob(*args, tau)
    tq, tk, tv, tdo = (torch.tensor(x, requires_grad=True) for x in args[:4])
    uq, uk, uv = (torch.tensor(x) for x in args[4:])
    out = torch.softmax(tau * tq @ tk.T, dim=-1) @ tv
    dq, dk, dv = torch.autograd.grad(out, (tq, tk, tv), tdo, create_graph=True)
    ph = (dq * uq).sum() + (dk * uk).sum() + (dv * uv).sum()
    g = torch.autograd.grad(ph, (tq, tk, tv, tdo))
    for key, t in zip(("dQt", "dKt", "dVt", "ddOt"), g):
        assert rel(r[key], t.numpy()) < 1e-12, key


def test_golden_fixture():
    """Stored oracle outputs (written by tests/golden/make_golden.py) guard
    against an unintended change of the oracle's arithmetic."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "bob_N6_d3_seed5.txt")
    data = {}
    with open(path) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            data[key] = np.array([float(v) for v in vals])
    args = rand_inputs(6, 3, 5)
    r = orc.bob(*args, 0.5)
    for key in ("dQt", "dKt", "dVt", "ddOt", "alpha", "E"):
        assert rel(r[key].ravel(), data[key]) < 1e-14, key


# --------------------------------------------------------------------------
# Causal mask (the setting of the pages' timing tables)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("N,d,seed", [(6, 3, 30), (11, 4, 31)])
def test_causal_bob_matches_fd_of_phi(N, d, seed):
    Q, K, V, dO, UQ, UK, UV = rand_inputs(N, d, seed)
    tau = 0.6
    r = orc.bob(Q, K, V, dO, UQ, UK, UV, tau, causal=True)
    args = [Q, K, V, dO]
    for pos, key in enumerate(("dQt", "dKt", "dVt", "ddOt")):
        def f(X, pos=pos):
            a = list(args)
            a[pos] = X
            return orc.phi(*a, UQ, UK, UV, tau, causal=True)
        assert rel(r[key], _fd_grad(f, args[pos])) < RTOL_FD, key


def test_causal_matches_bruteforce_rows_affine_and_torch():
    torch = pytest.importorskip("torch")
    N, d = 13, 5
    args = rand_inputs(N, d, 32)
    tau = 0.45
    r = orc.bob(*args, tau, causal=True)
    b = orc.bob_bruteforce(*args, tau, causal=True)
    a = orc.bob_affine(*args, tau, causal=True)
    rows = [0, 1, 6, 12]
    s = orc.bob_rows(*args, tau, rows, causal=True)
    for key in ("dQt", "dKt", "dVt", "ddOt", "alpha", "E"):
        assert rel(r[key], b[key]) < 1e-12, key
    for key in ("dQt", "ddOt", "alpha", "E"):
        assert rel(a[key], r[key]) < 1e-12, key
        assert rel(s[key], r[key][rows]) < 1e-12, key
    tq, tk, tv, tdo = (torch.tensor(x, requires_grad=True) for x in args[:4])
    uq, uk, uv = (torch.tensor(x) for x in args[4:])
    mask = torch.ones(N, N, dtype=torch.bool).tril()
    sc = (tau * tq @ tk.T).masked_fill(~mask, float("-inf"))
    out = torch.softmax(sc, dim=-1) @ tv
    dq, dk, dv = torch.autograd.grad(out, (tq, tk, tv), tdo, create_graph=True)
    ph = (dq * uq).sum() + (dk * uk).sum() + (dv * uv).sum()
    g = torch.autograd.grad(ph, (tq, tk, tv, tdo))
    for key, t in zip(("dQt", "dKt", "dVt", "ddOt"), g):
        assert rel(r[key], t.numpy()) < 1e-12, key


def test_causal_first_row_and_invariants():
    Q, K, V, dO, UQ, UK, UV = rand_inputs(9, 4, 33)
    tau = 0.5
    r = orc.bob(Q, K, V, dO, UQ, UK, UV, tau, causal=True)
    # query 0 sees only key 0: the N = 1 closed form for its row
    alpha0 = tau * (UQ[0] @ K[0] + Q[0] @ UK[0])
    assert np.isclose(r["alpha"][0], alpha0, rtol=1e-13)
    assert np.allclose(r["ddOt"][0], UV[0], rtol=1e-13, atol=1e-14)
    assert np.abs(r["dQt"][0]).max() < 1e-14
    # the last key is seen only by the last query: its softmax weight sits in
    # one row, and the shift invariances still hold
    ph = orc.phi(Q, K, V, dO, UQ, UK, UV, tau, causal=True)
    assert abs((r["ddOt"] * dO).sum() - ph) < 1e-12 * (abs(ph) + 1)
    assert np.abs(r["dKt"].sum(axis=0)).max() < 1e-12 * np.abs(r["dKt"]).max() * 9
    assert np.abs(r["dVt"].sum(axis=0)).max() < 1e-12 * np.abs(r["dVt"]).max() * 9


# --------------------------------------------------------------------------
# Grouped-query attention
# --------------------------------------------------------------------------

def _rand_gqa(H, Hkv, N, d, seed):
    rng = np.random.default_rng(seed)
    q = [rng.standard_normal((H, N, d)) for _ in range(2)]
    k = [rng.standard_normal((Hkv, N, d)) for _ in range(2)]
    dO, UQ = rng.standard_normal((H, N, d)), rng.standard_normal((H, N, d))
    UK, UV = rng.standard_normal((Hkv, N, d)), rng.standard_normal((Hkv, N, d))
    return q[0], k[0], k[1], dO, UQ, UK, UV


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_matches_fd_of_phi(causal):
    Q, K, V, dO, UQ, UK, UV = _rand_gqa(4, 2, 5, 3, 40)
    tau = 0.55
    r = orc.bob_gqa(Q, K, V, dO, UQ, UK, UV, tau, causal)
    args = [Q, K, V, dO]
    for pos, key in enumerate(("dQt", "dKt", "dVt", "ddOt")):
        def f(X, pos=pos):
            a = list(args)
            a[pos] = X
            return orc.phi_gqa(*a, UQ, UK, UV, tau, causal)
        assert rel(r[key], _fd_grad(f, args[pos])) < RTOL_FD, key


def test_gqa_matches_torch_double_backward_with_shared_heads():
    torch = pytest.importorskip("torch")
    H, Hkv, N, d = 6, 2, 9, 4
    Q, K, V, dO, UQ, UK, UV = _rand_gqa(H, Hkv, N, d, 41)
    tau = 0.5
    r = orc.bob_gqa(Q, K, V, dO, UQ, UK, UV, tau)
    tq, tk, tv, tdo = (torch.tensor(x, requires_grad=True) for x in (Q, K, V, dO))
    uq, uk, uv = (torch.tensor(x) for x in (UQ, UK, UV))
    kr = tk.repeat_interleave(H // Hkv, dim=0)  # autograd sums the group's gradients
    vr = tv.repeat_interleave(H // Hkv, dim=0)
    out = torch.softmax(tau * tq @ kr.transpose(1, 2), dim=-1) @ vr
    dq, dk, dv = torch.autograd.grad(out, (tq, tk, tv), tdo, create_graph=True)
    ph = (dq * uq).sum() + (dk * uk).sum() + (dv * uv).sum()
    g = torch.autograd.grad(ph, (tq, tk, tv, tdo))
    for key, t in zip(("dQt", "dKt", "dVt", "ddOt"), g):
        assert rel(r[key], t.numpy()) < 1e-12, key


def test_gqa_with_one_group_is_mha():
    Q, K, V, dO, UQ, UK, UV = _rand_gqa(3, 3, 7, 4, 42)
    r = orc.bob_gqa(Q, K, V, dO, UQ, UK, UV, 0.4)
    for h in range(3):
        m = orc.bob(Q[h], K[h], V[h], dO[h], UQ[h], UK[h], UV[h], 0.4)
        for key in ("dQt", "dKt", "dVt", "ddOt", "alpha", "E"):
            assert rel(r[key][h], m[key]) < 1e-14, key


# --------------------------------------------------------------------------
# Rectangular attention (N_q query rows, N_k key rows)
# --------------------------------------------------------------------------

def _rand_rect(Nq, Nk, d, seed):
    rng = np.random.default_rng(seed)
    q = [rng.standard_normal((Nq, d)) for _ in range(3)]  # Q, dO, U_Q
    k = [rng.standard_normal((Nk, d)) for _ in range(4)]  # K, V, U_K, U_V
    return q[0], k[0], k[1], q[1], q[2], k[2], k[3]


@pytest.mark.parametrize("Nq,Nk,causal", [(4, 9, False), (9, 4, False), (5, 8, True),
                                          (8, 5, True)])
def test_rectangular_bob_matches_fd_of_phi(Nq, Nk, causal):
    Q, K, V, dO, UQ, UK, UV = _rand_rect(Nq, Nk, 3, 50 + Nq)
    tau = 0.45
    r = orc.bob(Q, K, V, dO, UQ, UK, UV, tau, causal)
    assert r["dQt"].shape == (Nq, 3) and r["dKt"].shape == (Nk, 3)
    args = [Q, K, V, dO]
    for pos, key in enumerate(("dQt", "dKt", "dVt", "ddOt")):
        def f(X, pos=pos):
            a = list(args)
            a[pos] = X
            return orc.phi(*a, UQ, UK, UV, tau, causal)
        assert rel(r[key], _fd_grad(f, args[pos])) < RTOL_FD, key


@pytest.mark.parametrize("causal", [False, True])
def test_rectangular_matches_bruteforce_rows_affine_and_torch(causal):
    torch = pytest.importorskip("torch")
    Nq, Nk, d = 11, 7, 4
    args = _rand_rect(Nq, Nk, d, 51)
    tau = 0.5
    r = orc.bob(*args, tau, causal)
    b = orc.bob_bruteforce(*args, tau, causal)
    a = orc.bob_affine(*args, tau, causal)
    rows = [0, 3, 6, 7, 10]
    s = orc.bob_rows(*args, tau, rows, causal=causal)
    for key in ("dQt", "dKt", "dVt", "ddOt", "alpha", "E"):
        assert rel(r[key], b[key]) < 1e-12, key
    for key in ("dQt", "ddOt", "alpha", "E"):
        assert rel(a[key], r[key]) < 1e-12, key
        assert rel(s[key], r[key][rows]) < 1e-12, key
    # torch fp64 autograd double-backward, mask on absolute positions (j <= i)
    tq, tk, tv, tdo = (torch.tensor(x, requires_grad=True) for x in (args[0], args[1], args[2],
                                                                      args[3]))
    uq, uk, uv = (torch.tensor(x) for x in args[4:])
    sc = tau * tq @ tk.T
    if causal:
        keep = torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None]
        sc = sc.masked_fill(~keep, float("-inf"))
    out = torch.softmax(sc, dim=-1) @ tv
    dq, dk, dv = torch.autograd.grad(out, (tq, tk, tv), tdo, create_graph=True)
    ph = (dq * uq).sum() + (dk * uk).sum() + (dv * uv).sum()
    g = torch.autograd.grad(ph, (tq, tk, tv, tdo))
    for key, t in zip(("dQt", "dKt", "dVt", "ddOt"), g):
        assert rel(r[key], t.numpy()) < 1e-12, key


def test_rectangular_causal_unseen_keys_and_invariants():
    """Keys j >= N_q are seen by no query under the causal mask: their d~K,
    d~V are exactly zero; the shift invariances hold over the key axis."""
    Nq, Nk, d = 5, 9, 3
    Q, K, V, dO, UQ, UK, UV = _rand_rect(Nq, Nk, d, 52)
    r = orc.bob(Q, K, V, dO, UQ, UK, UV, 0.7, causal=True)
    assert np.abs(r["dKt"][Nq:]).max() == 0.0 and np.abs(r["dVt"][Nq:]).max() == 0.0
    for causal in (False, True):
        r = orc.bob(Q, K, V, dO, UQ, UK, UV, 0.7, causal=causal)
        ph = orc.phi(Q, K, V, dO, UQ, UK, UV, 0.7, causal=causal)
        assert abs((r["ddOt"] * dO).sum() - ph) < 1e-12 * (abs(ph) + 1)
        for key in ("dKt", "dVt"):
            assert np.abs(r[key].sum(axis=0)).max() < 1e-12 * np.abs(r[key]).max() * Nk


# --------------------------------------------------------------------------
# Attention JVP (forward-mode derivative along U_Q, U_K, U_V)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("Nq,Nk,causal", [(9, 9, False), (9, 9, True), (5, 11, True),
                                          (11, 5, False)])
def test_attention_jvp_matches_fd_of_the_forward(Nq, Nk, causal):
    Q, K, V, _, UQ, UK, UV = _rand_rect(Nq, Nk, 4, 60 + Nq + Nk)
    tau = 0.45
    O, L, Od, Ld = orc.attention_jvp(Q, K, V, UQ, UK, UV, tau, causal)
    h = 1e-5
    _, _, Op, Lp = orc.forward(Q + h * UQ, K + h * UK, V + h * UV, tau, causal)
    _, _, Om, Lm = orc.forward(Q - h * UQ, K - h * UK, V - h * UV, tau, causal)
    assert rel(Od, (Op - Om) / (2 * h)) < 1e-8
    assert rel(Ld, (Lp - Lm) / (2 * h)) < 1e-8
    _, _, O0, L0 = orc.forward(Q, K, V, tau, causal)
    assert rel(O, O0) < 1e-15 and rel(L, L0) < 1e-15


def test_attention_jvp_matches_torch_forward_ad():
    torch = pytest.importorskip("torch")
    import torch.autograd.forward_ad as fwAD
    Nq, Nk, d = 7, 10, 3
    Q, K, V, _, UQ, UK, UV = _rand_rect(Nq, Nk, d, 61)
    tau = 0.6
    for causal in (False, True):
        O, L, Od, Ld = orc.attention_jvp(Q, K, V, UQ, UK, UV, tau, causal)
        with fwAD.dual_level():
            q = fwAD.make_dual(torch.tensor(Q), torch.tensor(UQ))
            k = fwAD.make_dual(torch.tensor(K), torch.tensor(UK))
            v = fwAD.make_dual(torch.tensor(V), torch.tensor(UV))
            sc = tau * q @ k.T
            if causal:
                keep = torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None]
                sc = sc.masked_fill(~keep, float("-inf"))
            lse = torch.logsumexp(sc, dim=-1)
            out = torch.softmax(sc, dim=-1) @ v
            t_od = fwAD.unpack_dual(out).tangent.numpy()
            t_ld = fwAD.unpack_dual(lse).tangent.numpy()
        assert rel(Od, t_od) < 1e-12 and rel(Ld, t_ld) < 1e-12


def test_attention_jvp_is_the_bob_by_product():
    """alpha and d~dO of the BoB equal L' and O' for any dO."""
    Q, K, V, dO, UQ, UK, UV = _rand_rect(8, 12, 4, 62)
    _, _, Od, Ld = orc.attention_jvp(Q, K, V, UQ, UK, UV, 0.5, True)
    for scale in (1.0, -3.0):
        r = orc.bob(Q, K, V, scale * dO, UQ, UK, UV, 0.5, True)
        assert rel(r["ddOt"], Od) < 1e-13 and rel(r["alpha"], Ld) < 1e-13


# --------------------------------------------------------------------------
# Column form (d~K_j, d~V_j of chosen key columns) and the all-row scalars
# --------------------------------------------------------------------------

def _fd_entry(fun, X, idx, h=1e-5):
    Xp, Xm = X.copy(), X.copy()
    Xp[idx] += h
    Xm[idx] -= h
    return (fun(Xp) - fun(Xm)) / (2 * h)


@pytest.mark.parametrize("Nq,Nk,causal", [(9, 9, False), (9, 9, True), (6, 11, False),
                                          (11, 6, True)])
def test_bob_cols_matches_fd_of_phi(Nq, Nk, causal):
    """Each d~K_jk, d~V_jk of the column form is the derivative of Phi with
    respect to K_jk, V_jk (central differences, straight from the definition
    of Phi)."""
    rng = np.random.default_rng(50 + Nq + Nk)
    Q, dO, UQ = (rng.standard_normal((Nq, 4)) for _ in range(3))
    K, V, UK, UV = (rng.standard_normal((Nk, 4)) for _ in range(4))
    tau = 0.6
    cols = [0, Nk // 2, Nk - 1]
    r = orc.bob_cols(Q, K, V, dO, UQ, UK, UV, tau, cols, causal)
    for n, j in enumerate(cols):
        for k in range(4):
            fk = _fd_entry(lambda X: orc.phi(Q, X, V, dO, UQ, UK, UV, tau, causal), K, (j, k))
            fv = _fd_entry(lambda X: orc.phi(Q, K, X, dO, UQ, UK, UV, tau, causal), V, (j, k))
            assert abs(r["dKt"][n, k] - fk) <= 1e-7 * max(1.0, abs(fk)), (j, k)
            assert abs(r["dVt"][n, k] - fv) <= 1e-7 * max(1.0, abs(fv)), (j, k)


@pytest.mark.parametrize("causal", [False, True])
def test_bob_cols_matches_torch_double_backward(causal):
    torch = pytest.importorskip("torch")
    Nq, Nk, d = 13, 21, 5
    rng = np.random.default_rng(60)
    Q, dO, UQ = (rng.standard_normal((Nq, d)) for _ in range(3))
    K, V, UK, UV = (rng.standard_normal((Nk, d)) for _ in range(4))
    tau = 1 / np.sqrt(d)
    cols = np.array([0, 3, 12, 20])
    r = orc.bob_cols(Q, K, V, dO, UQ, UK, UV, tau, cols, causal)
    tq, tk, tv, tdo = (torch.tensor(x, requires_grad=True) for x in (Q, K, V, dO))
    uq, uk, uv = (torch.tensor(x) for x in (UQ, UK, UV))
    s = tau * tq @ tk.T
    if causal:
        s = s.masked_fill(~torch.tensor(orc.causal_mask(Nq, Nk)), float("-inf"))
    out = torch.softmax(s, dim=-1) @ tv
    dq, dk, dv = torch.autograd.grad(out, (tq, tk, tv), tdo, create_graph=True)
    ph = (dq * uq).sum() + (dk * uk).sum() + (dv * uv).sum()
    gk, gv = torch.autograd.grad(ph, (tk, tv))
    assert rel(r["dKt"], gk.numpy()[cols]) < 1e-12
    assert rel(r["dVt"], gv.numpy()[cols]) < 1e-12


@pytest.mark.parametrize("Nq,Nk,causal", [(40, 40, False), (40, 40, True), (25, 70, True),
                                          (70, 25, False)])
def test_row_scalars_and_bob_cols_match_matrix_form(Nq, Nk, causal):
    """Chunked all-row scalars and the column form against ``bob`` (whose
    pins are finite differences, sympy and torch); the chunk size splits the
    rows unevenly so that the ragged last chunk is covered."""
    rng = np.random.default_rng(70 + Nq)
    Q, dO, UQ = (rng.standard_normal((Nq, 8)) for _ in range(3))
    K, V, UK, UV = (rng.standard_normal((Nk, 8)) for _ in range(4))
    tau = 0.4
    full = orc.bob(Q, K, V, dO, UQ, UK, UV, tau, causal)
    sc = orc.row_scalars(Q, K, V, dO, UQ, UK, UV, tau, causal, chunk=7)
    for key in ("L", "D", "alpha", "E"):
        assert rel(sc[key], full[key]) < 1e-13, key
    cols = np.arange(Nk)
    r = orc.bob_cols(Q, K, V, dO, UQ, UK, UV, tau, cols, causal, scalars=sc)
    assert rel(r["dKt"], full["dKt"]) < 1e-13
    assert rel(r["dVt"], full["dVt"]) < 1e-13


def test_row_scalars_alpha_is_the_jvp_of_L():
    """alpha_i is the directional derivative of L_i along (U_Q, U_K) (finite
    differences of the forward), independently of ``bob``."""
    rng = np.random.default_rng(80)
    Q, K, V, dO, UQ, UK, UV = (rng.standard_normal((30, 6)) for _ in range(7))
    tau, h = 0.45, 1e-5
    sc = orc.row_scalars(Q, K, V, dO, UQ, UK, UV, tau, chunk=8)
    _, _, O, Lp = orc.forward(Q + h * UQ, K + h * UK, V, tau)
    _, _, _, Lm = orc.forward(Q - h * UQ, K - h * UK, V, tau)
    assert rel(sc["alpha"], (Lp - Lm) / (2 * h)) < 1e-8
    from scipy.special import logsumexp
    assert rel(sc["L"], logsumexp(tau * Q @ K.T, axis=1)) < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_bob_cols_group_matches_fd_of_phi_gqa(causal):
    Q, K, V, dO, UQ, UK, UV = _rand_gqa(4, 2, 6, 3, 90)
    tau = 0.55
    cols = [1, 4]
    for g in range(2):
        hs = slice(2 * g, 2 * g + 2)
        r = orc.bob_cols_group(Q[hs], K[g], V[g], dO[hs], UQ[hs], UK[g], UV[g], tau, cols,
                               causal)
        for n, j in enumerate(cols):
            for k in range(3):
                fk = _fd_entry(lambda X: orc.phi_gqa(Q, X, V, dO, UQ, UK, UV, tau, causal), K,
                               (g, j, k))
                fv = _fd_entry(lambda X: orc.phi_gqa(Q, K, X, dO, UQ, UK, UV, tau, causal), V,
                               (g, j, k))
                assert abs(r["dKt"][n, k] - fk) <= 1e-7 * max(1.0, abs(fk))
                assert abs(r["dVt"][n, k] - fv) <= 1e-7 * max(1.0, abs(fv))


def test_bob_batched_matches_torch_double_backward_over_batch_and_heads():
    """The [B, H] loop of ``bob_batched`` (every head, and a listed subset)
    against torch fp64 double-backward of Phi summed over all (b, h)."""
    torch = pytest.importorskip("torch")
    B, H, N, d = 2, 3, 10, 4
    rng = np.random.default_rng(95)
    args = [rng.standard_normal((B, H, N, d)) for _ in range(7)]
    tau = 0.5
    r = orc.bob_batched(*args, tau)
    tq, tk, tv, tdo = (torch.tensor(x, requires_grad=True) for x in args[:4])
    uq, uk, uv = (torch.tensor(x) for x in args[4:])
    out = torch.softmax(tau * tq @ tk.transpose(-1, -2), dim=-1) @ tv
    dq, dk, dv = torch.autograd.grad(out, (tq, tk, tv), tdo, create_graph=True)
    ph = (dq * uq).sum() + (dk * uk).sum() + (dv * uv).sum()
    g = torch.autograd.grad(ph, (tq, tk, tv, tdo))
    for key, t in zip(("dQt", "dKt", "dVt", "ddOt"), g):
        assert rel(r[key], t.numpy()) < 1e-12, key
    sub = orc.bob_batched(*args, tau, heads=[(1, 2), (0, 1)])
    for key, t in zip(("dQt", "dKt", "dVt", "ddOt"), g):
        for b, h in ((1, 2), (0, 1)):
            assert rel(sub[key][b, h], t.numpy()[b, h]) < 1e-12, key
        assert np.isnan(sub[key][0, 0]).all()  # heads not listed stay unwritten


@pytest.mark.parametrize("Nq,Nk,causal", [(1, 1, False), (33, 33, False), (65, 65, True),
                                          (70, 25, True), (25, 70, True), (100, 3, False)])
def test_c_row_scalars_match_numpy_and_matrix_form(Nq, Nk, causal):
    """The plain-C row scalars (oracle/rowscal.c) against ``bob`` and the
    numpy ``row_scalars``, on shapes whose row count is not a multiple of the
    C code's 32-row groups; inputs are fp32-exact (bf16-rounded) values."""
    torch = pytest.importorskip("torch")
    from oracle import crows
    rng = np.random.default_rng(100 + Nq + Nk)
    q = [torch.tensor(rng.standard_normal((Nq, 7))).to(torch.bfloat16).double().numpy()
         for _ in range(3)]
    k = [torch.tensor(rng.standard_normal((Nk, 7))).to(torch.bfloat16).double().numpy()
         for _ in range(4)]
    Q, dO, UQ = q
    K, V, UK, UV = k
    tau = 0.42
    c = crows.row_scalars(Q, K, V, dO, UQ, UK, UV, tau, causal)
    full = orc.bob(Q, K, V, dO, UQ, UK, UV, tau, causal)
    for key in ("L", "D", "alpha", "E"):
        assert rel(c[key], full[key]) < 1e-13, key


def test_c_row_scalars_rejects_inexact_inputs():
    from oracle import crows
    x = np.full((4, 3), 0.1)  # 0.1 is not an fp32 value
    with pytest.raises(ValueError):
        crows.row_scalars(x, x, x, x, x, x, x, 0.5)


@pytest.mark.parametrize("Nq,Nk,causal,scale", [(23, 23, False, 1.0), (23, 23, True, 1.0),
                                                (9, 31, False, 2.0), (31, 9, True, 0.5)])
def test_E_is_the_row_dot_of_dO_and_ddOt(Nq, Nk, causal, scale):
    # E_i = sum_j P_ij d~P_ij with d~P = F o (dP - D) + G - alpha dP expands,
    # through dP = dO V^T, G = dO U_V^T and D = dO . O, into the row dot
    # dO_i . d~dO_i - alpha_i D_i (d~dO = P U_V + P o (F - alpha) V): E and
    # d~dO come from different parts of the chain rule (the softmax node and
    # the dO node), so this ties the two together.
    Q, K, V, dO, UQ, UK, UV = [scale * m for m in _rand_rect(Nq, Nk, 5, 70 + Nq + Nk)]
    r = orc.bob(Q, K, V, dO, UQ, UK, UV, 0.4, causal=causal)
    E2 = (dO * r["ddOt"]).sum(axis=1) - r["alpha"] * r["D"]
    assert np.allclose(E2, r["E"], rtol=1e-12, atol=1e-12 * np.abs(r["E"]).max())
