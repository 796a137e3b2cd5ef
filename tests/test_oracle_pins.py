"""Pins for the float64 CPU oracle: checks against things other than itself.

Each test ties the oracle to what the Gaussian Mixture Attention pages fix
(gist.science technical summaries, "Core mechanism" items 1-2, "Variants and
training" item 3) or to mathematics / library routines that do not share its
code:

* scipy.stats.multivariate_normal densities for the GMM posterior;
* scipy.spatial.distance + scipy.special.softmax for the isotropic case;
* the materialised affinity A = Gamma_Q Gamma_K^T (and its lower triangle)
  for the bidirectional and causal outputs on tiny N;
* closed forms (K = 1 means, hand-derived 1-d examples in tests/golden/);
* invariants (permutations, prior shift, mass conservation, convex hull,
  rank <= K).

The backward pass (gradients given dL/dO; "Variants and training" item 3:
the components are learned by backpropagation) is pinned by central finite
differences of the forward oracle, element by element.

Cross-attention (N queries reading the memory of Nk keys; gist.science
summary, "Significance and claims": cross-attention named as future work) is
pinned the same way: the materialised N x Nk affinity, the K = 1 mean, no
keys, and key-permutation invariance.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats
from scipy.spatial.distance import cdist

from gaussian_mixture_sequence_gma_gb300.inputs import make_inputs, make_params
from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "gmm_posterior_1d.txt")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _small_problem(seed, B=1, H=2, N=24, d=6, dv=3, K=5, smin=0.1):
    r = _rng(seed)
    Q = r.standard_normal((B, H, N, d))
    Kx = r.standard_normal((B, H, N, d))
    V = r.standard_normal((B, H, N, dv))
    mu = r.standard_normal((H, K, d))
    sigma2 = np.log1p(np.exp(r.standard_normal((H, K, d)))) + smin
    log_pi = np.log(scipy.special.softmax(r.standard_normal((H, K)), axis=-1))
    return Q, Kx, V, mu, sigma2, log_pi


def _scipy_gamma(X, mu, sigma2, log_pi):
    """Posterior via scipy's multivariate normal log-density (independent code)."""
    B, H, N, d = X.shape
    K = mu.shape[1]
    G = np.empty((B, H, N, K))
    for b in range(B):
        for h in range(H):
            lp = np.stack([scipy.stats.multivariate_normal(mean=mu[h, k], cov=np.diag(sigma2[h, k])).logpdf(X[b, h])
                           for k in range(K)], axis=-1).reshape(N, K)
            G[b, h] = scipy.special.softmax(lp + log_pi[h][None, :], axis=-1)
    return G


def _brute(Q, Kx, V, mu, sigma2, log_pi, eps, causal):
    GQ = _scipy_gamma(Q, mu, sigma2, log_pi)
    GK = _scipy_gamma(Kx, mu, sigma2, log_pi)
    A = np.einsum("bhik,bhjk->bhij", GQ, GK)
    if causal:
        A = np.tril(A)
    num = np.einsum("bhij,bhjc->bhic", A, V)
    den = A.sum(-1, keepdims=True) + eps
    return num / den


# ----------------------------------------------------------------------------- Gamma

@pytest.mark.parametrize("K,sig", [(16, 1.0), (128, 0.5), (256, 1.0)])
def test_gamma_rows_are_distributions(K, sig):
    inp = make_inputs(1, 2, 300, K, dtype="f32", seed=11, sigma_raw_std=sig)
    G = orc.responsibilities(inp["Q"], inp["mu"], inp["sigma2"], inp["log_pi"])
    assert G.min() >= 0.0
    assert np.abs(G.sum(-1) - 1.0).max() <= 1e-12


def test_gamma_matches_explicit_density_ratio():
    # pi_k N(x; mu_k, Sigma_k) / sum_j pi_j N(x; mu_j, Sigma_j) with explicit pdfs, small d (no underflow).
    Q, _, _, mu, sigma2, log_pi = _small_problem(1, d=4, K=6, smin=0.3)
    G = orc.responsibilities(Q, mu, sigma2, log_pi)
    B, H, N, d = Q.shape
    for h in range(H):
        dens = np.stack([np.exp(log_pi[h, k]) * scipy.stats.multivariate_normal(mu[h, k], np.diag(sigma2[h, k])).pdf(Q[0, h])
                         for k in range(mu.shape[1])], axis=-1)
        ref = dens / dens.sum(-1, keepdims=True)
        assert np.abs(G[0, h] - ref).max() <= 1e-12


def test_gamma_d64_matches_scipy_logpdf():
    inp = make_inputs(1, 2, 64, 16, dtype="f32", seed=5, sigma_raw_std=1.0)
    G = orc.responsibilities(inp["Q"], inp["mu"], inp["sigma2"], inp["log_pi"])
    ref = _scipy_gamma(inp["Q"].astype(np.float64), inp["mu"].astype(np.float64), inp["sigma2"].astype(np.float64),
                       inp["log_pi"].astype(np.float64))
    assert np.abs(G - ref).max() <= 1e-11


def test_gamma_isotropic_uniform_is_softmax_of_distances():
    r = _rng(3)
    N, K, d, s2 = 40, 7, 5, 0.8
    X = r.standard_normal((1, 1, N, d))
    mu = r.standard_normal((1, K, d))
    sigma2 = np.full((1, K, d), s2)
    log_pi = np.full((1, K), -math.log(K))
    G = orc.responsibilities(X, mu, sigma2, log_pi)
    ref = scipy.special.softmax(-cdist(X[0, 0], mu[0], "sqeuclidean") / (2 * s2), axis=-1)
    assert np.abs(G[0, 0] - ref).max() <= 1e-12


def test_gamma_invariant_to_prior_shift_and_component_order():
    Q, _, _, mu, sigma2, log_pi = _small_problem(4, K=7)
    G = orc.responsibilities(Q, mu, sigma2, log_pi)
    G2 = orc.responsibilities(Q, mu, sigma2, log_pi + 3.25)
    assert np.abs(G - G2).max() <= 1e-12
    perm = _rng(9).permutation(mu.shape[1])
    G3 = orc.responsibilities(Q, mu[:, perm], sigma2[:, perm], log_pi[:, perm])
    assert np.abs(G[..., perm] - G3).max() <= 1e-12


def test_gamma_row_sampling_matches_full():
    Q, _, _, mu, sigma2, log_pi = _small_problem(6, N=50)
    G = orc.responsibilities(Q, mu, sigma2, log_pi)
    rows = [0, 7, 49]
    assert np.array_equal(orc.responsibilities(Q, mu, sigma2, log_pi, rows=rows), G[:, :, rows])


# ----------------------------------------------------------------------------- forward vs brute force

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("eps", [1e-6, 0.37])
def test_forward_matches_materialised_affinity(causal, eps):
    Q, Kx, V, mu, sigma2, log_pi = _small_problem(7, B=2, H=2, N=33, d=6, dv=3, K=5)
    O = orc.forward(Q, Kx, V, mu, sigma2, log_pi, eps, causal=causal)
    ref = _brute(Q, Kx, V, mu, sigma2, log_pi, eps, causal)
    assert np.abs(O - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


@pytest.mark.parametrize("causal", [False, True])
def test_forward_d64_matches_materialised_affinity(causal):
    inp = make_inputs(1, 1, 40, 16, dtype="f32", seed=8, sigma_raw_std=1.0)
    args = [inp[k].astype(np.float64) for k in ("Q", "K", "V", "mu", "sigma2", "log_pi")]
    O = orc.forward(*args, 1e-6, causal=causal)
    ref = _brute(*args, 1e-6, causal)
    assert np.abs(O - ref).max() <= 1e-11 * np.abs(ref).max()


@pytest.mark.parametrize("causal", [False, True])
def test_forward_row_sampling_matches_full(causal):
    Q, Kx, V, mu, sigma2, log_pi = _small_problem(12, N=40)
    O = orc.forward(Q, Kx, V, mu, sigma2, log_pi, 1e-6, causal=causal)
    rows = [0, 1, 17, 39]
    Os = orc.forward(Q, Kx, V, mu, sigma2, log_pi, 1e-6, causal=causal, rows=rows)
    assert np.array_equal(Os, O[:, :, rows])


# ----------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("eps", [1e-6, 0.5])
def test_single_component_is_mean_and_running_mean(eps):
    r = _rng(13)
    N, d, dv = 29, 4, 3
    Q = r.standard_normal((1, 1, N, d)); Kx = r.standard_normal((1, 1, N, d)); V = r.standard_normal((1, 1, N, dv))
    mu = r.standard_normal((1, 1, d)); sigma2 = np.full((1, 1, d), 0.7); log_pi = np.zeros((1, 1))
    Ob = orc.forward(Q, Kx, V, mu, sigma2, log_pi, eps, causal=False)[0, 0]
    assert np.abs(Ob - V[0, 0].sum(0) / (N + eps)).max() <= 1e-13
    Oc = orc.forward(Q, Kx, V, mu, sigma2, log_pi, eps, causal=True)[0, 0]
    run = np.cumsum(V[0, 0], axis=0) / (np.arange(1, N + 1)[:, None] + eps)
    assert np.abs(Oc - run).max() <= 1e-13


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or "|" not in line:
                continue
            k, v = line.split("|")
            vals[k.strip()] = np.array([float(x) for x in v.split(",")])
    return vals


def test_golden_worked_examples():
    g = _golden()
    a = math.log(3.0) / 2
    mu = np.array([[[-1.0], [1.0]]]); s2 = np.ones((1, 2, 1)); lp = np.log(np.full((1, 2), 0.5))
    X = np.array([a, -a, 0.0]).reshape(1, 1, 3, 1)
    G = orc.responsibilities(X, mu, s2, lp)[0, 0]
    assert np.abs(G[0] - g["caseA.gamma_at_a"]).max() < 1e-15
    assert np.abs(G[1] - g["caseA.gamma_at_minus_a"]).max() < 1e-15
    assert np.abs(G[2] - g["caseA.gamma_at_0"]).max() < 1e-15
    Kx = np.array([-a, a]).reshape(1, 1, 2, 1); V = np.array([1.0, 3.0]).reshape(1, 1, 2, 1)
    Vt, Z = orc.state(Kx, V, mu, s2, lp)
    assert np.abs(Vt[0, 0, :, 0] - g["caseA.state_Vt"]).max() < 1e-14
    assert np.abs(Z[0, 0] - g["caseA.state_Z"]).max() < 1e-14
    Q0 = np.zeros((1, 1, 2, 1))
    assert abs(orc.forward(Q0, Kx, V, mu, s2, lp, 0.0)[0, 0, 0, 0] - g["caseA.bidir_O_q0_eps0"][0]) < 1e-14
    assert abs(orc.forward(Q0, Kx, V, mu, s2, lp, 0.5)[0, 0, 0, 0] - g["caseA.bidir_O_q0_eps0.5"][0]) < 1e-14
    assert abs(orc.forward(Kx, Kx, V, mu, s2, lp, 0.0)[0, 0, 0, 0] - g["caseA.bidir_O_qminusa_eps0"][0]) < 1e-14
    assert np.abs(orc.forward(Kx, Kx, V, mu, s2, lp, 0.0, causal=True)[0, 0, :, 0] - g["caseA.causal_O_eps0"]).max() < 1e-14
    assert np.abs(orc.forward(Kx, Kx, V, mu, s2, lp, 0.25, causal=True)[0, 0, :, 0]
                  - g["caseA.causal_O_eps0.25"]).max() < 1e-14
    # case B: log-determinant term
    mu = np.zeros((1, 2, 1)); s2 = np.array([1.0, 4.0]).reshape(1, 2, 1)
    b = math.sqrt(8 * math.log(2) / 3)
    G = orc.responsibilities(np.array([0.0, b]).reshape(1, 1, 2, 1), mu, s2, lp)[0, 0]
    assert abs(G[0, 0] - g["caseB.gamma1_at_0"][0]) < 1e-15
    assert abs(G[1, 0] - g["caseB.gamma1_at_b"][0]) < 1e-15


# ----------------------------------------------------------------------------- invariants

def test_output_invariant_to_component_permutation():
    Q, Kx, V, mu, sigma2, log_pi = _small_problem(14, N=30, K=6)
    perm = _rng(1).permutation(6)
    for causal in (False, True):
        O = orc.forward(Q, Kx, V, mu, sigma2, log_pi, 1e-3, causal=causal)
        O2 = orc.forward(Q, Kx, V, mu[:, perm], sigma2[:, perm], log_pi[:, perm], 1e-3, causal=causal)
        assert np.abs(O - O2).max() <= 1e-12


def test_bidir_token_permutation_equivariance():
    Q, Kx, V, mu, sigma2, log_pi = _small_problem(15, N=31)
    r = _rng(2)
    pq = r.permutation(31)
    pk = r.permutation(31)
    O = orc.forward(Q, Kx, V, mu, sigma2, log_pi, 1e-3)
    O2 = orc.forward(Q[:, :, pq], Kx[:, :, pk], V[:, :, pk], mu, sigma2, log_pi, 1e-3)
    assert np.abs(O[:, :, pq] - O2).max() <= 1e-12


def test_state_mass_and_brute_state():
    Q, Kx, V, mu, sigma2, log_pi = _small_problem(16, N=45, K=4)
    Vt, Z = orc.state(Kx, V, mu, sigma2, log_pi)
    assert np.abs(Z.sum(-1) - 45).max() <= 1e-12
    GK = _scipy_gamma(Kx, mu, sigma2, log_pi)
    assert np.abs(Vt - np.einsum("bhjk,bhjc->bhkc", GK, V)).max() <= 1e-12


def test_outputs_in_convex_hull_of_values():
    inp = make_inputs(1, 2, 200, 16, dtype="f32", seed=17)
    for causal in (False, True):
        O = orc.forward(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 0.0, causal=causal)
        V = inp["V"].astype(np.float64)
        if causal:
            lo = np.minimum.accumulate(V, axis=2); hi = np.maximum.accumulate(V, axis=2)
        else:
            lo = V.min(2, keepdims=True); hi = V.max(2, keepdims=True)
        assert (O >= lo - 1e-12).all() and (O <= hi + 1e-12).all()


def test_affinity_rank_at_most_K():
    Q, Kx, V, mu, sigma2, log_pi = _small_problem(18, N=40, K=5, d=3)
    GQ = orc.responsibilities(Q, mu, sigma2, log_pi)[0, 0]
    GK = orc.responsibilities(Kx, mu, sigma2, log_pi)[0, 0]
    A = GQ @ GK.T
    assert A.min() >= 0
    assert np.linalg.matrix_rank(A, tol=1e-10) <= 5


def test_causal_endpoints():
    Q, Kx, V, mu, sigma2, log_pi = _small_problem(19, N=26)
    eps = 0.2
    Ob = orc.forward(Q, Kx, V, mu, sigma2, log_pi, eps)
    Oc = orc.forward(Q, Kx, V, mu, sigma2, log_pi, eps, causal=True)
    assert np.abs(Ob[:, :, -1] - Oc[:, :, -1]).max() <= 1e-12
    GQ = orc.responsibilities(Q, mu, sigma2, log_pi)
    GK = orc.responsibilities(Kx, mu, sigma2, log_pi)
    g = (GQ[:, :, 0] * GK[:, :, 0]).sum(-1)[..., None]
    assert np.abs(Oc[:, :, 0] - V[:, :, 0] * g / (g + eps)).max() <= 1e-12


# ----------------------------------------------------------------------------- cross-attention

def _brute_cross(Q, Kx, V, mu, sigma2, log_pi, eps):
    GQ = _scipy_gamma(Q, mu, sigma2, log_pi)
    GK = _scipy_gamma(Kx, mu, sigma2, log_pi)
    A = np.einsum("bhik,bhjk->bhij", GQ, GK)  # N x Nk
    return np.einsum("bhij,bhjc->bhic", A, V) / (A.sum(-1, keepdims=True) + eps)


def _cross_problem(seed, N, Nk, B=2, H=2, d=5, dv=3, K=4):
    Q, _, _, mu, sigma2, log_pi = _small_problem(seed, B=B, H=H, N=N, d=d, dv=dv, K=K, smin=0.3)
    r = _rng(seed + 1000)
    Kx = r.standard_normal((B, H, Nk, d))
    V = r.standard_normal((B, H, Nk, dv))
    return Q, Kx, V, mu, sigma2, log_pi


@pytest.mark.parametrize("N,Nk,eps", [(17, 29, 1e-6), (31, 5, 0.37), (1, 40, 1e-6)])
def test_cross_matches_materialised_affinity(N, Nk, eps):
    Q, Kx, V, mu, sigma2, log_pi = _cross_problem(5, N, Nk)
    O = orc.forward_cross(Q, Kx, V, mu, sigma2, log_pi, eps)
    ref = _brute_cross(Q, Kx, V, mu, sigma2, log_pi, eps)
    assert O.shape == ref.shape
    assert np.abs(O - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


@pytest.mark.parametrize("eps", [1e-6, 0.5])
def test_cross_single_component_is_key_mean(eps):
    # K = 1: every gamma is 1, so every query reads sum_j v_j / (Nk + eps)
    Q, Kx, V, mu, sigma2, log_pi = _cross_problem(7, 9, 23, K=1)
    O = orc.forward_cross(Q, Kx, V, mu, sigma2, log_pi, eps)
    want = V.sum(2, keepdims=True) / (23 + eps)
    assert np.abs(O - np.broadcast_to(want, O.shape)).max() <= 1e-13


def test_cross_without_keys_is_zero():
    Q, Kx, V, mu, sigma2, log_pi = _cross_problem(8, 6, 0)
    O = orc.forward_cross(Q, Kx, V, mu, sigma2, log_pi, 1e-6)
    assert O.shape == (2, 2, 6, 3) and np.all(O == 0.0)


def test_cross_key_permutation_invariance():
    Q, Kx, V, mu, sigma2, log_pi = _cross_problem(9, 12, 19)
    perm = _rng(3).permutation(19)
    O1 = orc.forward_cross(Q, Kx, V, mu, sigma2, log_pi, 1e-6)
    O2 = orc.forward_cross(Q, Kx[:, :, perm], V[:, :, perm], mu, sigma2, log_pi, 1e-6)
    assert np.abs(O1 - O2).max() <= 1e-12


# ----------------------------------------------------------------------------- backward

def _fd_grads(Q, Kx, V, mu, sigma2, log_pi, eps, G, h=1e-6, lib=None, causal=False):
    """Central finite differences of L = sum(O * G) through the forward oracle, every element."""
    args = [Q, Kx, V, mu, sigma2, log_pi]
    out = []
    for a in range(6):
        g = np.zeros_like(args[a])
        flat = g.reshape(-1)
        for idx in range(flat.size):
            vals = [x.copy() for x in args]
            step = h * max(1.0, abs(vals[a].reshape(-1)[idx]))
            vals[a].reshape(-1)[idx] += step
            lp = (orc.forward(*vals, eps, causal=causal, lib=lib) * G).sum()
            vals[a].reshape(-1)[idx] -= 2 * step
            lm = (orc.forward(*vals, eps, causal=causal, lib=lib) * G).sum()
            flat[idx] = (lp - lm) / (2 * step)
        out.append(g)
    return out


@pytest.mark.parametrize("eps", [1e-6, 0.37])
def test_backward_matches_finite_differences(eps):
    Q, Kx, V, mu, sigma2, log_pi = _small_problem(31, B=2, H=2, N=5, d=3, dv=2, K=3, smin=0.3)
    G = _rng(32).standard_normal((2, 2, 5, 2))
    got = orc.backward_bidir(Q, Kx, V, mu, sigma2, log_pi, eps, G)
    want = _fd_grads(Q, Kx, V, mu, sigma2, log_pi, eps, G)
    for name, a, b in zip(("dQ", "dK", "dV", "dmu", "dsigma2", "dlog_pi"), got, want):
        assert a.shape == b.shape, name
        assert np.abs(a - b).max() <= 1e-6 * max(1.0, np.abs(b).max()), name


@pytest.mark.parametrize("eps", [1e-6, 0.37])
def test_causal_backward_matches_finite_differences(eps):
    Q, Kx, V, mu, sigma2, log_pi = _small_problem(41, B=2, H=2, N=6, d=3, dv=2, K=3, smin=0.3)
    G = _rng(42).standard_normal((2, 2, 6, 2))
    got = orc.backward_causal(Q, Kx, V, mu, sigma2, log_pi, eps, G)
    want = _fd_grads(Q, Kx, V, mu, sigma2, log_pi, eps, G, causal=True)
    for name, a, b in zip(("dQ", "dK", "dV", "dmu", "dsigma2", "dlog_pi"), got, want):
        assert a.shape == b.shape, name
        assert np.abs(a - b).max() <= 1e-6 * max(1.0, np.abs(b).max()), name


def test_causal_backward_last_row_only_matches_bidir():
    # a loss on the last output alone: that row sees every key, as in the bidirectional form
    Q, Kx, V, mu, sigma2, log_pi = _small_problem(43, B=1, H=2, N=8, d=4, dv=3, K=4, smin=0.3)
    G = np.zeros((1, 2, 8, 3))
    G[:, :, -1] = _rng(44).standard_normal((1, 2, 3))
    c = orc.backward_causal(Q, Kx, V, mu, sigma2, log_pi, 1e-6, G)
    b = orc.backward_bidir(Q, Kx, V, mu, sigma2, log_pi, 1e-6, G)
    for x, y in zip(c, b):
        assert np.abs(x - y).max() <= 1e-12 * max(1.0, np.abs(y).max())


def test_backward_prior_gradient_sums_to_zero():
    # shifting every log pi_k of a head by the same constant leaves O unchanged
    Q, Kx, V, mu, sigma2, log_pi = _small_problem(33, B=1, H=2, N=9, d=4, dv=3, K=4, smin=0.3)
    G = _rng(34).standard_normal((1, 2, 9, 3))
    dlp = orc.backward_bidir(Q, Kx, V, mu, sigma2, log_pi, 1e-6, G)[5]
    assert np.abs(dlp.sum(-1)).max() <= 1e-12 * max(1.0, np.abs(dlp).max())


def test_backward_values_gradient_is_linear_read():
    # O is linear in V: dV_j = sum_i G_i A_ij / den_i with the materialised affinity
    Q, Kx, V, mu, sigma2, log_pi = _small_problem(35, B=1, H=1, N=7, d=4, dv=3, K=3, smin=0.3)
    G = _rng(36).standard_normal((1, 1, 7, 3))
    eps = 0.2
    GQ, GK = _scipy_gamma(Q, mu, sigma2, log_pi), _scipy_gamma(Kx, mu, sigma2, log_pi)
    A = np.einsum("bhik,bhjk->bhij", GQ, GK)
    den = A.sum(-1, keepdims=True) + eps
    want = np.einsum("bhij,bhic->bhjc", A / den, G)
    dV = orc.backward_bidir(Q, Kx, V, mu, sigma2, log_pi, eps, G)[2]
    assert np.abs(dV - want).max() <= 1e-12 * max(1.0, np.abs(want).max())


# ----------------------------------------------------------------------------- planted mistakes

MUTANTS = {
    "drop_logdet": ("- 0.5 * (quad + logdet[k])", "- 0.5 * (quad)"),
    "sign_flip": ("- 0.5 * (quad + logdet[k])", "+ 0.5 * (quad + logdet[k])"),
    "drop_prior": ("double l = log_pi[k]", "double l = 0.0 * log_pi[k]"),
    "drop_eps": ("den += J->eps;", "den += 0.0;"),
    "value_index": ("g[k] * V[(size_t)j * dv + c]", "g[k] * V[(size_t)j * dv + (dv - 1 - c)]"),
    "cross_key_stride": ("const double *Kx = J->Kx + (size_t)unit * Nk * d;",
                         "const double *Kx = J->Kx + (size_t)unit * N * d;"),
    "cross_write_over_queries": ("for (int j = 0; j < Nk; ++j) {", "for (int j = 0; j < N && j < Nk; ++j) {"),
    "bwd_drops_denominator_term": ("const double dden = -gdoto / den;", "const double dden = 0.0 * gdoto;"),
    "bwd_variance_sign": ("0.5 * (diff * diff / (s2 * s2) - 1.0 / s2)", "0.5 * (diff * diff / (s2 * s2) + 1.0 / s2)"),
    "bwd_causal_suffix_excludes_own_query": (
        "for (int c = 0; c < C; ++c) R[(size_t)k * C + c] += gqj[k] * uj[c];\n      for (int k = 0; k < K; ++k) {\n        double s = R[(size_t)k * C + dv];",
        "for (int c = 0; c < C; ++c) R[(size_t)k * C + c] += 0.0 * gqj[k] * uj[c];\n      for (int k = 0; k < K; ++k) {\n        double s = R[(size_t)k * C + dv];"),
    "bwd_softmax_no_centering": ("dl[k] = g[k] * (dg[k] - dot);", "dl[k] = g[k] * dg[k];"),
    "causal_drops_first_key": ("int64_t want = J->rows ? J->rows[r] : i;",
                         "int64_t want = J->rows ? J->rows[r] : i; if (i == 0) { memset(Vt, 0, sizeof(double) * K * dv); memset(Z, 0, sizeof(double) * K); }"),
}


def _pins_pass(lib) -> bool:
    """A compact subset of the pins above, run against a given oracle build."""
    try:
        Q, Kx, V, mu, sigma2, log_pi = _small_problem(21, N=20, d=4, dv=3, K=4, smin=0.3)
        for causal in (False, True):
            O = orc.forward(Q, Kx, V, mu, sigma2, log_pi, 0.37, causal=causal, lib=lib)
            if np.abs(O - _brute(Q, Kx, V, mu, sigma2, log_pi, 0.37, causal)).max() > 1e-10:
                return False
        G = orc.responsibilities(Q, mu, sigma2, log_pi, lib=lib)
        if np.abs(G - _scipy_gamma(Q, mu, sigma2, log_pi)).max() > 1e-10:
            return False
        Q, Kx, V, mu, sigma2, log_pi = _small_problem(23, B=1, H=2, N=4, d=2, dv=2, K=3, smin=0.3)
        G = _rng(24).standard_normal((1, 2, 4, 2))
        for causal in (False, True):
            got = orc.backward_bidir(Q, Kx, V, mu, sigma2, log_pi, 0.37, G, lib=lib, causal=causal)
            want = _fd_grads(Q, Kx, V, mu, sigma2, log_pi, 0.37, G, lib=lib, causal=causal)
            for a, b in zip(got, want):
                if np.abs(a - b).max() > 1e-6 * max(1.0, np.abs(b).max()):
                    return False
        Q, Kx, V, mu, sigma2, log_pi = _cross_problem(22, 7, 13)
        O = orc.forward_cross(Q, Kx, V, mu, sigma2, log_pi, 0.37, lib=lib)
        if np.abs(O - _brute_cross(Q, Kx, V, mu, sigma2, log_pi, 0.37)).max() > 1e-10:
            return False
        return True
    except Exception:
        return False


def test_pins_pass_on_the_real_oracle():
    assert _pins_pass(orc._load())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    src = open(orc._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, name
    mutated = src.replace(old, new)
    p = tmp_path / "mutant.c"
    p.write_text(mutated)
    so = orc.build(force=True, src=str(p), out=str(tmp_path / "libmutant.so"))
    assert not _pins_pass(orc._load(so)), "pins missed mutant %s" % name


# ----------------------------------------------------------------------------- projected (Transformer block)

def test_round_to_bf16_matches_torch():
    # pinned to an independent implementation of round-to-nearest-even bfloat16 (torch's conversion)
    torch = pytest.importorskip("torch")
    r = np.random.Generator(np.random.PCG64(3))
    x = np.concatenate([r.standard_normal(4096) * 10.0 ** r.integers(-6, 6, 4096),
                        [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -1.0 - 2.0 ** -8, 0.0, 65504.0]])
    ours = orc.round_to_bf16(x)
    theirs = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, theirs)
    assert orc.round_to_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 1.0  # a tie goes to the even neighbour


def test_projection_brute_force():
    r = np.random.Generator(np.random.PCG64(4))
    B, N, H, dm = 2, 3, 2, 5
    X = r.standard_normal((B, N, dm))
    W = r.standard_normal((dm, 3 * H * 64))
    b = r.standard_normal(3 * H * 64)
    Q, Kx, V = orc.project_qkv(X, W, b, H, "f32")
    for w, T in enumerate((Q, Kx, V)):
        for bb in range(B):
            for h in range(H):
                for n in range(N):
                    for dd in (0, 17, 63):
                        c = (w * H + h) * 64 + dd
                        want = sum(X[bb, n, m] * W[m, c] for m in range(dm)) + b[c]
                        assert abs(T[bb, h, n, dd] - want) < 1e-12


def test_projected_identity_weights_reduce_to_forward():
    r = np.random.Generator(np.random.PCG64(5))
    B, H, N, K = 1, 2, 40, 6
    X = r.standard_normal((B, N, H * 64))
    W = np.concatenate([np.eye(H * 64)] * 3, axis=1)
    mu = r.standard_normal((H, K, 64))
    sigma2 = 0.5 + r.random((H, K, 64))
    log_pi = np.log(np.full((H, K), 1.0 / K))
    Xh = np.ascontiguousarray(X.reshape(B, N, H, 64).transpose(0, 2, 1, 3))
    for causal in (False, True):
        got = orc.forward_projected(X, W, np.zeros(3 * H * 64), mu, sigma2, log_pi, 1e-6, causal=causal, dtype="f32")
        want = orc.forward(Xh, Xh, Xh, mu, sigma2, log_pi, 1e-6, causal=causal)
        assert np.allclose(got, want, rtol=0, atol=1e-12)
    # a transposed weight is a different projection (the identity above would not notice it)
    W2 = r.standard_normal((H * 64, 3 * H * 64)) / 8
    a = orc.forward_projected(X, W2, np.zeros(3 * H * 64), mu, sigma2, log_pi, 1e-6, dtype="f32")
    Wt = np.concatenate([W2[:, w * H * 64:(w + 1) * H * 64].T for w in range(3)], axis=1)
    b = orc.forward_projected(X, Wt, np.zeros(3 * H * 64), mu, sigma2, log_pi, 1e-6, dtype="f32")
    assert np.abs(a - b).max() > 1e-3
