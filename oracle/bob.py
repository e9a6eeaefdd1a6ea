"""Plain fp64 oracle for exact backward-over-backward of softmax attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``.  The CUDA library never imports,
links or calls it, and it shares no code with the CUDA path.

Every function works on ONE (batch, head) slice: 2-D numpy arrays in
float64 (rows are sequence positions), plus the scale ``tau``.  The query-side
arrays Q, dO, U_Q are ``[N_q, d]`` and the key-side arrays K, V, U_K, U_V are
``[N_k, d]``; N_q = N_k is ordinary self-attention, N_q != N_k rectangular
attention.  The batched helpers at the end loop over ``[B, H]``.

Sources (web pages on the method; sections named as on the pages):

* [FBN] "FlashBoB: I/O-Efficient Exact Backward-over-Backward for Softmax
  Attention", paper notes (papernotes.org): section 方法详解/整体框架 (the
  objective Phi and the four outputs) and 关键设计 1 (the row scalars D, alpha,
  E, the matrix F, the affine rule for d~P and the three affine corrections).
* [FAB] "FlashAttention 的反向传播设计：在 SRAM 内部重计算 Softmax 的显存收益"
  (bjdmk.com.cn): section 一 (forward S, P, O and the first backward dV, dP,
  dS, D, dQ, dK) and section 二 (recomputing P from saved row statistics).

Readings where the pages are silent (each is listed in the design notes):

* L is the natural-log logsumexp of the scaled scores, P = exp(S - L).
* D_i = dO_i . O_i, which equals sum_j P_ij dP_ij ([FAB] section 一).
* The pages print F, alpha, E, the d~P rule and the corrections, but not
  d~K, d~V, nor what B, R and Omega contain.  ``bob`` differentiates Phi by
  hand (chain rule through F, G, dP, D and the softmax); ``bob_affine`` then
  names B = P K, R = (P o dP) K, Omega = (P o d~P0) K + dS U_K, the only
  assignment that makes the printed corrections alpha-free and exact.

Parity pins (tests/test_oracle.py): central finite differences of Phi, exact
symbolic differentiation (sympy) on tiny inputs, a loop-only brute force,
the printed affine identities, sum_j P_ij = 1, shift invariances, Hessian
symmetry, the N = 1 closed form, the U_Q = U_K = 0 reduction to a first
backward, JVP identities of the forward and torch fp64 double-backward.  The
row form (``bob_rows``), the all-row scalars (``row_scalars``), the column
form (``bob_cols``, ``bob_cols_group``) and the batched loop
(``bob_batched``) each have pins of their own (finite differences of Phi
entry by entry, torch double-backward, the matrix form).  No function here
is unpinned.
"""
from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# Forward, row state and first backward  ([FAB] sections 一 and 二)
# --------------------------------------------------------------------------

def causal_mask(Nq, Nk=None):
    """True where key j is visible from query i (j <= i): the causal mask of
    the pages' benchmarks ([FBN] 实验关键数据).  For N_q != N_k the same
    rule on absolute positions (the mask's diagonal starts at the top left),
    so every query row sees at least key 0."""
    Nk = Nq if Nk is None else Nk
    return np.tril(np.ones((Nq, Nk), dtype=bool))


def forward(Q, K, V, tau, causal=False):
    """S = tau Q K^T, L = logsumexp_j S_ij, P = exp(S - L), O = P V.

    [FAB] section 一 (S, P = softmax(S), O = P V) with the softmax written
    through the saved row statistic L as in [FAB] section 二.  With
    ``causal`` the scores of keys j > i are -inf, so P_ij = 0 there.
    """
    S = tau * (Q @ K.T)
    if causal:
        S = np.where(causal_mask(Q.shape[0], K.shape[0]), S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    L = m[:, 0] + np.log(np.exp(S - m).sum(axis=1))
    P = np.exp(S - L[:, None])
    O = P @ V
    return S, P, O, L


def prep(Q, K, V, dO, tau, causal=False):
    """Row state the BoB consumes: O, L and D_i = dO_i . O_i.

    [FBN] 关键设计 1 defines D_i = dO_i^T O_i; [FAB] section 一 gives the same
    scalar as sum_j dP_ij P_ij.
    """
    _, _, O, L = forward(Q, K, V, tau, causal)
    D = (dO * O).sum(axis=1)
    return O, L, D


def first_backward(Q, K, V, dO, tau, causal=False):
    """dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = tau dS K, dK = tau dS^T Q.

    [FAB] section 一.  The 1/sqrt(d) of the page is the general scale tau.
    """
    _, P, O, _ = forward(Q, K, V, tau, causal)
    dV = P.T @ dO
    dP = dO @ V.T
    D = (P * dP).sum(axis=1)
    dS = P * (dP - D[:, None])
    dQ = tau * (dS @ K)
    dK = tau * (dS.T @ Q)
    return dQ, dK, dV


def phi(Q, K, V, dO, UQ, UK, UV, tau, causal=False):
    """Phi = <dQ, U_Q> + <dK, U_K> + <dV, U_V>  ([FBN] 方法详解/整体框架)."""
    dQ, dK, dV = first_backward(Q, K, V, dO, tau, causal)
    return float((dQ * UQ).sum() + (dK * UK).sum() + (dV * UV).sum())


# --------------------------------------------------------------------------
# Backward-over-backward, plain matrix form
# --------------------------------------------------------------------------

def bob(Q, K, V, dO, UQ, UK, UV, tau, causal=False):
    """Total derivatives of Phi w.r.t. Q, K, V and dO, with O, L, D functions
    of the inputs ([FBN] 方法详解/整体框架).

    Phi rewritten with the first backward: Phi = sum_ij dS_ij F_ij +
    sum_ij P_ij G_ij, where F = tau (U_Q K^T + Q U_K^T) ([FBN] 关键设计 1)
    and G = dO U_V^T.  Chain rule, one node at a time:

    * through D:   dPhi/dP_ij holds  d~P = d~P0 - alpha dP  with
      d~P0 = F o (dP - D) + G and alpha_i = sum_j P_ij F_ij  ([FBN] 关键设计 1);
    * through the softmax: d~S = P o (d~P - E), E_i = sum_j P_ij d~P_ij;
    * through dP = dO V^T: the gradient w.r.t. dP is P o (F - alpha);
    * through F and G: gradients dS and P.

    Returns d~Q = tau (d~S K + dS U_K), d~K = tau (d~S^T Q + dS^T U_Q),
    d~V = (P o (F - alpha))^T dO, d~dO = P U_V + (P o (F - alpha)) V,
    and the row scalars alpha and E.  With ``causal`` P vanishes above the
    diagonal, and every term above carries a factor P.
    """
    S, P, O, L = forward(Q, K, V, tau, causal)
    dP = dO @ V.T
    D = (dO * O).sum(axis=1)
    dS = P * (dP - D[:, None])
    F = tau * (UQ @ K.T + Q @ UK.T)
    G = dO @ UV.T
    alpha = (P * F).sum(axis=1)
    dPt0 = F * (dP - D[:, None]) + G
    dPt = dPt0 - alpha[:, None] * dP
    E = (P * dPt).sum(axis=1)
    dSt = P * (dPt - E[:, None])
    dPdP = P * (F - alpha[:, None])  # gradient of Phi w.r.t. dP
    return {
        "dQt": tau * (dSt @ K + dS @ UK),
        "dKt": tau * (dSt.T @ Q + dS.T @ UQ),
        "dVt": dPdP.T @ dO,
        "ddOt": P @ UV + dPdP @ V,
        "alpha": alpha,
        "E": E,
        "L": L,
        "D": D,
    }


def bob_affine(Q, K, V, dO, UQ, UK, UV, tau, causal=False):
    """Row outputs through the alpha-free accumulators and the affine
    correction of [FBN] 关键设计 1:

        E = E0 - alpha D,  d~dO = d~dO0 - alpha O,  d~Q = tau (Omega - alpha R - E B)

    with E0_i = sum_j P_ij d~P0_ij, B = P K, R = (P o dP) K,
    Omega = (P o d~P0) K + dS U_K and d~dO0 = P U_V + (P o F) V.
    """
    S, P, O, L = forward(Q, K, V, tau, causal)
    dP = dO @ V.T
    D = (dO * O).sum(axis=1)
    dS = P * (dP - D[:, None])
    F = tau * (UQ @ K.T + Q @ UK.T)
    G = dO @ UV.T
    dPt0 = F * (dP - D[:, None]) + G
    alpha = (P * F).sum(axis=1)
    E0 = (P * dPt0).sum(axis=1)
    B = P @ K
    R = (P * dP) @ K
    Omega = (P * dPt0) @ K + dS @ UK
    ddOt0 = P @ UV + (P * F) @ V
    E = E0 - alpha * D
    return {
        "dQt": tau * (Omega - alpha[:, None] * R - E[:, None] * B),
        "ddOt": ddOt0 - alpha[:, None] * O,
        "alpha": alpha,
        "E": E,
        "E0": E0,
    }


# --------------------------------------------------------------------------
# Forward-mode derivative of attention (the JVP by-product of pass 1)
# --------------------------------------------------------------------------

def attention_jvp(Q, K, V, UQ, UK, UV, tau, causal=False):
    """Directional derivative of the attention forward along (U_Q, U_K, U_V),
    by its definition: with S = tau Q K^T and its tangent
    S' = tau (U_Q K^T + Q U_K^T), the softmax tangent is
    P' = P o (S' - rowsum(P o S')), so that

        L' = rowsum(P o S'),   O' = P' V + P U_V.

    Returns (O, L, O', L').  S' is the matrix F of [FBN] 关键设计 1, and
    L', O' are the alpha and d~dO that pass 1 produces (reading them as a
    JVP is this module's reading; the pins check it against finite
    differences and torch forward-mode AD).
    """
    S, P, O, L = forward(Q, K, V, tau, causal)
    Sd = tau * (UQ @ K.T + Q @ UK.T)
    if causal:
        Sd = np.where(causal_mask(Q.shape[0], K.shape[0]), Sd, 0.0)
    Ld = (P * Sd).sum(axis=1)
    Pd = P * (Sd - Ld[:, None])
    Od = Pd @ V + P @ UV
    return O, L, Od, Ld


# --------------------------------------------------------------------------
# One row at a time: O(N d) per row, for long sequences
# --------------------------------------------------------------------------

def bob_rows(Q, K, V, dO, UQ, UK, UV, tau, rows, causal=False):
    """Row-side outputs (L, D, alpha, E, d~Q, d~dO) for the listed rows only.

    The same definitions as ``bob`` restricted to row i: every quantity of
    row i needs only row i of Q, dO, U_Q and all of K, V, U_K, U_V (only the
    keys j <= i with ``causal``).
    """
    rows = np.asarray(rows, dtype=np.int64)
    out = {k: [] for k in ("L", "D", "alpha", "E", "dQt", "ddOt")}
    for i in rows:
        s = tau * (K @ Q[i])
        if causal:
            s = np.where(np.arange(K.shape[0]) <= i, s, -np.inf)
        m = s.max()
        Li = m + np.log(np.exp(s - m).sum())
        p = np.exp(s - Li)
        o = p @ V
        Di = dO[i] @ o
        dp = V @ dO[i]
        ds = p * (dp - Di)
        f = tau * (K @ UQ[i] + UK @ Q[i])
        g = UV @ dO[i]
        a = p @ f
        dpt = f * (dp - Di) + g - a * dp
        Ei = p @ dpt
        dst = p * (dpt - Ei)
        out["L"].append(Li)
        out["D"].append(Di)
        out["alpha"].append(a)
        out["E"].append(Ei)
        out["dQt"].append(tau * (dst @ K + ds @ UK))
        out["ddOt"].append(p @ UV + (p * (f - a)) @ V)
    return {k: np.array(v) for k, v in out.items()}


# --------------------------------------------------------------------------
# One key column at a time: the column outputs d~K_j, d~V_j for long sequences
# --------------------------------------------------------------------------

def row_scalars(Q, K, V, dO, UQ, UK, UV, tau, causal=False, chunk=256):
    """L, D, alpha and E of every query row, by the same definitions as
    ``bob`` ([FAB] sections 一/二 for L and D, [FBN] 关键设计 1 for alpha and
    E), evaluated for ``chunk`` rows at a time so that no N_q x N_k array is
    held at once.  The rows are independent: each row's values are exactly
    those ``bob`` computes for it."""
    Nq = Q.shape[0]
    L, D, alpha, E = (np.empty(Nq) for _ in range(4))
    for r0 in range(0, Nq, chunk):
        r = slice(r0, min(Nq, r0 + chunk))
        S = tau * (Q[r] @ K.T)
        if causal:
            S = np.where(causal_mask(Nq, K.shape[0])[r], S, -np.inf)
        m = S.max(axis=1, keepdims=True)
        Lr = m[:, 0] + np.log(np.exp(S - m).sum(axis=1))
        P = np.exp(S - Lr[:, None])
        Dr = (dO[r] * (P @ V)).sum(axis=1)
        F = tau * (UQ[r] @ K.T + Q[r] @ UK.T)
        dP = dO[r] @ V.T
        G = dO[r] @ UV.T
        ar = (P * F).sum(axis=1)
        dPt = F * (dP - Dr[:, None]) + G - ar[:, None] * dP
        L[r], D[r], alpha[r], E[r] = Lr, Dr, ar, (P * dPt).sum(axis=1)
    return {"L": L, "D": D, "alpha": alpha, "E": E}


def bob_cols(Q, K, V, dO, UQ, UK, UV, tau, cols, causal=False, scalars=None, chunk=64):
    """Column outputs d~K_j and d~V_j for the listed key columns j only.

    Column j of the transposed scores needs K_j, V_j, U_K,j, U_V,j, every
    query-side row and the row scalars L, D, alpha, E of every row ([FBN]
    关键设计 2: those scalars are all that crosses from the row pass to the
    column pass).  Given them, each column costs O(N_q d):

        P_ij = exp(tau Q_i.K_j - L_i),  dP_ij = dO_i.V_j,
        F_ij = tau (U_Q,i.K_j + Q_i.U_K,j),  G_ij = dO_i.U_V,j,
        dS = P (dP - D),  d~P = F (dP - D) + G - alpha dP,  d~S = P (d~P - E),
        d~K_j = tau sum_i (d~S_ij Q_i + dS_ij U_Q,i),
        d~V_j = sum_i P_ij (F_ij - alpha_i) dO_i

    (the formulas of ``bob`` read down one column), for ``chunk`` listed
    columns at a time.  ``scalars`` is a dict with L, D, alpha, E from
    ``row_scalars`` or ``bob``; when omitted they are computed here with
    ``row_scalars`` (O(N_q N_k d)).
    """
    sc = scalars if scalars is not None else row_scalars(Q, K, V, dO, UQ, UK, UV, tau, causal)
    L, D, alpha, E = (sc[k][:, None] for k in ("L", "D", "alpha", "E"))
    cols = np.asarray(cols, dtype=np.int64)
    d = Q.shape[1]
    dKt = np.empty((cols.size, d))
    dVt = np.empty((cols.size, d))
    rows = np.arange(Q.shape[0])[:, None]
    for c0 in range(0, cols.size, chunk):
        c = cols[c0:c0 + chunk]
        S = tau * (Q @ K[c].T)  # [N_q, columns]
        if causal:
            S = np.where(rows >= c[None, :], S, -np.inf)
        P = np.exp(S - L)
        dP = dO @ V[c].T
        F = tau * (UQ @ K[c].T + Q @ UK[c].T)
        G = dO @ UV[c].T
        dS = P * (dP - D)
        dPt = F * (dP - D) + G - alpha * dP
        dSt = P * (dPt - E)
        dKt[c0:c0 + c.size] = tau * (dSt.T @ Q + dS.T @ UQ)
        dVt[c0:c0 + c.size] = (P * (F - alpha)).T @ dO
    return {"dKt": dKt, "dVt": dVt}


def bob_cols_group(Qg, K, V, dOg, UQg, UK, UV, tau, cols, causal=False, scalars=None):
    """``bob_cols`` for a key/value head shared by the query heads of a group
    (``Qg``, ``dOg``, ``UQg`` are [G, N_q, d]): d~K_j, d~V_j of the shared
    head are the sums of the per-query-head columns ([FBN] 关键设计 3).
    ``scalars``, if given, is a list of one dict per query head."""
    out = {"dKt": 0.0, "dVt": 0.0}
    for h in range(Qg.shape[0]):
        r = bob_cols(Qg[h], K, V, dOg[h], UQg[h], UK, UV, tau, cols, causal,
                     None if scalars is None else scalars[h])
        out["dKt"] = out["dKt"] + r["dKt"]
        out["dVt"] = out["dVt"] + r["dVt"]
    return out


# --------------------------------------------------------------------------
# Brute force: scalar loops only (tiny N, d), an independent restatement
# --------------------------------------------------------------------------

def bob_bruteforce(Q, K, V, dO, UQ, UK, UV, tau, causal=False):
    """The same derivatives as ``bob`` written as explicit element sums.

    No matrix products, no vectorised reductions: every entry is a nested
    loop over (i, j, k), so a transposed operand or a dropped term in the
    matrix form shows up as a mismatch.
    """
    Nq, d = Q.shape
    Nk = K.shape[0]

    def dot(a, b):
        s = 0.0
        for k in range(d):
            s += a[k] * b[k]
        return s

    def visible(i, j):
        return j <= i or not causal

    S = [[tau * dot(Q[i], K[j]) for j in range(Nk)] for i in range(Nq)]
    P = [[0.0] * Nk for _ in range(Nq)]
    L = [0.0] * Nq
    for i in range(Nq):
        m = max(S[i][j] for j in range(Nk) if visible(i, j))
        z = 0.0
        for j in range(Nk):
            if visible(i, j):
                z += np.exp(S[i][j] - m)
        L[i] = m + np.log(z)
        for j in range(Nk):
            P[i][j] = np.exp(S[i][j] - L[i]) if visible(i, j) else 0.0
    O = [[sum(P[i][j] * V[j][k] for j in range(Nk)) for k in range(d)] for i in range(Nq)]
    D = [dot(dO[i], O[i]) for i in range(Nq)]
    dP = [[dot(dO[i], V[j]) for j in range(Nk)] for i in range(Nq)]
    F = [[tau * (dot(UQ[i], K[j]) + dot(Q[i], UK[j])) for j in range(Nk)] for i in range(Nq)]
    G = [[dot(dO[i], UV[j]) for j in range(Nk)] for i in range(Nq)]
    alpha = [sum(P[i][j] * F[i][j] for j in range(Nk)) for i in range(Nq)]
    dPt = [[F[i][j] * (dP[i][j] - D[i]) + G[i][j] - alpha[i] * dP[i][j] for j in range(Nk)]
           for i in range(Nq)]
    E = [sum(P[i][j] * dPt[i][j] for j in range(Nk)) for i in range(Nq)]
    dS = [[P[i][j] * (dP[i][j] - D[i]) for j in range(Nk)] for i in range(Nq)]
    dSt = [[P[i][j] * (dPt[i][j] - E[i]) for j in range(Nk)] for i in range(Nq)]
    dQt = np.zeros((Nq, d))
    dKt = np.zeros((Nk, d))
    dVt = np.zeros((Nk, d))
    ddOt = np.zeros((Nq, d))
    for i in range(Nq):
        for j in range(Nk):
            w = P[i][j] * (F[i][j] - alpha[i])
            for k in range(d):
                dQt[i, k] += tau * (dSt[i][j] * K[j][k] + dS[i][j] * UK[j][k])
                dKt[j, k] += tau * (dSt[i][j] * Q[i][k] + dS[i][j] * UQ[i][k])
                dVt[j, k] += w * dO[i][k]
                ddOt[i, k] += P[i][j] * UV[j][k] + w * V[j][k]
    return {"dQt": dQt, "dKt": dKt, "dVt": dVt, "ddOt": ddOt,
            "alpha": np.array(alpha), "E": np.array(E)}


# --------------------------------------------------------------------------
# Batched helpers over [B, H, N, d]
# --------------------------------------------------------------------------

def bob_batched(Q, K, V, dO, UQ, UK, UV, tau, heads=None, causal=False):
    """``bob`` for every (b, h) (or the listed (b, h) pairs)."""
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    shapes = {"dQt": (B, H, Nq, d), "ddOt": (B, H, Nq, d), "dKt": (B, H, Nk, d),
              "dVt": (B, H, Nk, d)}
    keys = ("dQt", "dKt", "dVt", "ddOt", "alpha", "E", "L", "D")
    out = {k: np.full(shapes.get(k, (B, H, Nq)), np.nan) for k in keys}
    pairs = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pairs:
        r = bob(Q[b, h], K[b, h], V[b, h], dO[b, h], UQ[b, h], UK[b, h], UV[b, h], tau, causal)
        for k in keys:
            out[k][b, h] = r[k]
    return out


# --------------------------------------------------------------------------
# Grouped-query attention: H query heads share H_kv key/value heads
# --------------------------------------------------------------------------

def phi_gqa(Q, K, V, dO, UQ, UK, UV, tau, causal=False):
    """Phi for [H, N_q, d] query-side arrays and [H_kv, N_k, d] key-side arrays:
    query head h attends to key/value head h // (H / H_kv), and the first
    backward's dK, dV of a shared head sum the contributions of its query
    heads ([FBN] 关键设计 3), so Phi is the sum of the per-head objectives."""
    H, Hkv = Q.shape[0], K.shape[0]
    G = H // Hkv
    total = 0.0
    for h in range(H):
        g = h // G
        total += phi(Q[h], K[g], V[g], dO[h], UQ[h], UK[g], UV[g], tau, causal)
    return total


def bob_gqa(Q, K, V, dO, UQ, UK, UV, tau, causal=False):
    """BoB of ``phi_gqa``: d~Q, d~dO, alpha, E per query head; d~K, d~V of a
    shared head are the sums over its query heads of the per-head results."""
    H, Hkv = Q.shape[0], K.shape[0]
    G = H // Hkv
    out = {"dQt": np.zeros(Q.shape), "ddOt": np.zeros(Q.shape), "dKt": np.zeros(K.shape),
           "dVt": np.zeros(K.shape), "alpha": np.zeros(Q.shape[:2]), "E": np.zeros(Q.shape[:2]),
           "L": np.zeros(Q.shape[:2]), "D": np.zeros(Q.shape[:2])}
    for h in range(H):
        g = h // G
        r = bob(Q[h], K[g], V[g], dO[h], UQ[h], UK[g], UV[g], tau, causal)
        for k in ("dQt", "ddOt", "alpha", "E", "L", "D"):
            out[k][h] = r[k]
        out["dKt"][g] += r["dKt"]
        out["dVt"][g] += r["dVt"]
    return out
