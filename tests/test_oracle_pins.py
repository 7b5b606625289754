"""Pins of the fp64 oracle against things other than itself.

Each test ties one step of the oracle to a closed form, a library routine, a
brute-force computation written independently here, an invariant, or the
hand-derived example in tests/golden/hand_example.txt. The steps are those of
"MiTA Attention: Efficient Fast-Weight Scaling via a Mixture of Top-k
Activations" (gist.science summaries: Arabic edition section 2 for pooling,
shared expert and top-k sets; Dutch edition "Wiskundige Formulering" for the
concatenated K* / V*; "Complexiteit" for the O(N(m + ks)) cost).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- pooling

@pytest.mark.parametrize("N,m", [(64, 8), (100, 7), (33, 33), (10, 1), (1000, 16)])
def test_pool_1d_matches_torch_adaptive_avg_pool(N, m):
    Q = _rand((2, N, 5), 1)
    got = oracle.pool(Q, m)
    ref = torch.nn.functional.adaptive_avg_pool1d(torch.from_numpy(Q).transpose(1, 2), m)
    np.testing.assert_allclose(got, ref.transpose(1, 2).numpy(), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("gh,gw,lh,lw", [(16, 16, 4, 4), (12, 10, 5, 3), (8, 8, 8, 8), (6, 9, 1, 2)])
def test_pool_2d_matches_torch_adaptive_avg_pool(gh, gw, lh, lw):
    d = 3
    Q = _rand((1, gh * gw, d), 2)
    got = oracle.pool(Q, lh * lw, grid=(gh, gw), lm=(lh, lw))
    img = torch.from_numpy(Q[0]).reshape(gh, gw, d).permute(2, 0, 1)[None]
    ref = torch.nn.functional.adaptive_avg_pool2d(img, (lh, lw))[0].permute(1, 2, 0).reshape(lh * lw, d)
    np.testing.assert_allclose(got[0], ref.numpy(), rtol=1e-13, atol=1e-13)


def test_pool_divisible_is_window_mean():
    Q = _rand((1, 96, 4), 3)
    np.testing.assert_allclose(oracle.pool(Q, 12)[0], Q[0].reshape(12, 8, 4).mean(axis=1), rtol=1e-13)


# -------------------------------------------------------- hand example

def _golden():
    vals = {}
    with open(os.path.join(GOLDEN, "hand_example.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, *rest = line.split()
            vals[name] = np.array([float(x) for x in rest])
    return vals


def test_hand_example():
    g = _golden()
    Q = np.array([0.0, 0.0, 1.0, 1.0]).reshape(1, 4, 1)
    K = np.array([0.0, 0.0, math.log(3.0), 0.0]).reshape(1, 4, 1)
    V = np.array([1.0, 2.0, 3.0, 4.0]).reshape(1, 4, 1)
    r = oracle.forward(Q, K, V, m=2, k=1, s=1, scale=1.0, threads=1)
    np.testing.assert_allclose(r["Qt"].ravel(), g["Qt"], rtol=1e-15)
    np.testing.assert_allclose(r["Vt"].ravel(), g["Vt"], rtol=1e-14)
    np.testing.assert_array_equal(r["I"].ravel(), g["I"].astype(int))
    np.testing.assert_array_equal(r["E"].ravel(), g["E"].astype(int))
    np.testing.assert_allclose(r["O"].ravel(), g["O"], rtol=1e-14)


# ------------------------------------------------------------ raw scores
# oracle.scores supplies every raw score the parity rules judge (top-k sets on
# k_j . qt_i, routes on q . qt_i), so it is pinned on its own.

@pytest.mark.parametrize("na,nb,d", [(7, 13, 5), (1, 40, 128), (33, 2, 64)])
def test_scores_match_numpy_matmul(na, nb, d):
    A, B = _rand((na, d), 11), _rand((nb, d), 12)
    got = oracle.scores(A, B)
    assert got.shape == (na, nb)
    np.testing.assert_allclose(got, A @ B.T, rtol=1e-12, atol=1e-12)


def test_scores_exact_on_integers():
    # small-integer inputs: every product and sum is exact in float64, so the
    # scores must equal the int64 matrix product exactly
    rng = np.random.default_rng(13)
    A = rng.integers(-50, 51, size=(9, 31))
    B = rng.integers(-50, 51, size=(17, 31))
    np.testing.assert_array_equal(oracle.scores(A.astype(np.float64), B.astype(np.float64)), (A @ B.T).astype(np.float64))


def test_scores_orientation():
    # A = unit rows e_c picks coordinate c of every row of B: S = B^T
    d, nb = 6, 10
    B = _rand((nb, d), 14)
    np.testing.assert_array_equal(oracle.scores(np.eye(d), B), B.T)
    np.testing.assert_array_equal(oracle.scores(B, np.eye(d)), B)


# ------------------------------------------------------ top-k and routing

def _brute_topk(S, k):
    """First k column indices of each row by (score desc, index asc), ascending."""
    out = []
    for row in S:
        order = np.lexsort((np.arange(len(row)), -row))
        out.append(np.sort(order[:k]))
    return np.array(out)


def _brute_route(R, s):
    return np.array([np.lexsort((np.arange(len(r)), -r))[:s] for r in R])


@pytest.mark.parametrize("N,d,m,k,s", [(200, 8, 5, 17, 2), (64, 4, 4, 64, 3), (50, 3, 10, 1, 1)])
def test_topk_and_routes_match_brute_force(N, d, m, k, s):
    rng = np.random.default_rng(5)
    Q, K, V = (rng.standard_normal((2, N, d)) for _ in range(3))
    r = oracle.forward(Q, K, V, m=m, k=k, s=s, threads=2)
    for h in range(2):
        Qt = Q[h].reshape(m, -1, d).mean(axis=1) if N % m == 0 else r["Qt"][h]
        np.testing.assert_allclose(r["Qt"][h], Qt, rtol=1e-12, atol=1e-14)
        np.testing.assert_array_equal(r["I"][h], _brute_topk(r["Qt"][h] @ K[h].T, k))
        np.testing.assert_array_equal(r["E"][h], _brute_route(Q[h] @ r["Qt"][h].T, s))


def test_topk_ties_go_to_lower_index():
    # keys take 3 values only, so every score row is full of exact ties
    rng = np.random.default_rng(7)
    N, d, m, k = 120, 2, 4, 30
    K = rng.integers(-1, 2, size=(1, N, d)).astype(np.float64)
    Q = rng.integers(-1, 2, size=(1, N, d)).astype(np.float64)
    V = rng.standard_normal((1, N, d))
    r = oracle.forward(Q, K, V, m=m, k=k, s=2, threads=1)
    S = r["Qt"][0] @ K[0].T
    np.testing.assert_array_equal(r["I"][0], _brute_topk(S, k))
    np.testing.assert_array_equal(r["E"][0], _brute_route(Q[0] @ r["Qt"][0].T, 2))


def test_negative_zero_ties_with_zero():
    # score rows of +0.0 and -0.0 are all equal: the lowest indices must win
    N, d = 16, 1
    K = np.zeros((1, N, d)); K[0, ::2, 0] = -0.0
    Q = np.ones((1, N, d))
    r = oracle.forward(Q, K, np.ones((1, N, d)), m=2, k=5, s=1, threads=1)
    np.testing.assert_array_equal(r["I"][0], np.tile(np.arange(5), (2, 1)))


# ------------------------------------------------ special-case identities

def _sdpa(q, k, v, scale):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None]
    return torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), scale=scale)[0].numpy()


@pytest.mark.parametrize("scale", [0.0, 0.37])
def test_no_shared_full_k_is_softmax_attention(scale):
    N, d = 48, 6
    Q, K, V = (_rand((1, N, d), i) for i in (10, 11, 12))
    r = oracle.forward(Q, K, V, m=4, k=N, s=1, scale=scale, no_shared=True, threads=1)
    tau = scale if scale > 0 else 1 / math.sqrt(d)
    np.testing.assert_allclose(r["O"][0], _sdpa(Q[0], K[0], V[0], tau), rtol=1e-12, atol=1e-13)


def test_shared_full_k_is_attention_over_landmarks_and_keys():
    N, d, m = 40, 5, 8
    Q, K, V = (_rand((1, N, d), i) for i in (20, 21, 22))
    r = oracle.forward(Q, K, V, m=m, k=N, s=1, threads=1)
    tau = 1 / math.sqrt(d)
    Qt = torch.nn.functional.adaptive_avg_pool1d(torch.from_numpy(Q[0]).T[None], m)[0].T.numpy()
    Vt = _sdpa(Qt, K[0], V[0], tau)
    np.testing.assert_allclose(r["Vt"][0], Vt, rtol=1e-12, atol=1e-13)
    ref = _sdpa(Q[0], np.concatenate([Qt, K[0]]), np.concatenate([Vt, V[0]]), tau)
    np.testing.assert_allclose(r["O"][0], ref, rtol=1e-12, atol=1e-13)


def test_overlapping_experts_are_concatenated():
    # all landmarks equal -> both experts hold every key -> each key is in two
    # slots, i.e. its logit carries an extra ln 2 against the shared slots
    N, d = 32, 4
    q = _rand((1, 1, d), 30)
    Q = np.repeat(q, N, axis=1)
    K, V = _rand((1, N, d), 31), _rand((1, N, d), 32)
    r = oracle.forward(Q, K, V, m=2, k=N, s=2, threads=1)
    np.testing.assert_array_equal(r["E"][0], np.tile([0, 1], (N, 1)))
    tau = 1 / math.sqrt(d)
    keys = np.concatenate([r["Qt"][0], K[0]])
    vals = np.concatenate([r["Vt"][0], V[0]])
    logits = tau * q[0] @ keys.T
    logits[:, 2:] += math.log(2.0)
    w = np.exp(logits - logits.max())
    ref = (w @ vals) / w.sum()
    np.testing.assert_allclose(r["O"][0], np.repeat(ref, N, axis=0), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------- invariants

def test_joint_key_value_permutation():
    N, d, m, k, s = 96, 6, 6, 11, 2
    Q, K, V = (_rand((1, N, d), i) for i in (40, 41, 42))
    perm = np.random.default_rng(43).permutation(N)
    a = oracle.forward(Q, K, V, m=m, k=k, s=s, threads=1)
    b = oracle.forward(Q, K[:, perm], V[:, perm], m=m, k=k, s=s, threads=1)
    # key j of the permuted input is original key perm[j]
    np.testing.assert_array_equal(np.sort(perm[b["I"][0]], axis=1), a["I"][0])
    np.testing.assert_allclose(b["O"], a["O"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["Vt"], a["Vt"], rtol=1e-12, atol=1e-13)


def test_outputs_in_convex_hull():
    N, d, m, k, s = 128, 8, 8, 16, 3
    Q, K, V = (_rand((1, N, d), i) for i in (50, 51, 52))
    r = oracle.forward(Q, K, V, m=m, k=k, s=s, threads=1)
    lo, hi = V[0].min(axis=0), V[0].max(axis=0)
    assert np.all(r["Vt"][0] >= lo - 1e-12) and np.all(r["Vt"][0] <= hi + 1e-12)
    vstar = np.concatenate([r["Vt"][0], V[0]])
    assert np.all(r["O"][0] >= vstar.min(axis=0) - 1e-12)
    assert np.all(r["O"][0] <= vstar.max(axis=0) + 1e-12)


def test_operation_count_is_linear_in_N():
    # multiply-adds: 2mNd (scores + Vt), Nmd (routing), 2N(m + sk)d (output)
    for N, d, m, k, s in [(64, 4, 4, 8, 2), (256, 8, 16, 32, 3), (512, 2, 8, 5, 1)]:
        Q, K, V = (_rand((1, N, d), i) for i in (60, 61, 62))
        r = oracle.forward(Q, K, V, m=m, k=k, s=s, threads=1)
        assert r["macs"] == 5 * N * m * d + 2 * N * s * k * d


def test_query_subset_and_overrides_reproduce_full_run():
    N, d, m, k, s = 80, 5, 5, 9, 2
    Q, K, V = (_rand((2, N, d), i) for i in (70, 71, 72))
    full = oracle.forward(Q, K, V, m=m, k=k, s=s, threads=2)
    ids = np.array([3, 79, 0, 41])
    sub = oracle.forward(Q, K, V, m=m, k=k, s=s, q_ids=ids, threads=2)
    np.testing.assert_array_equal(sub["E"], full["E"][:, ids])
    np.testing.assert_allclose(sub["O"], full["O"][:, ids], rtol=0, atol=0)
    ov = oracle.forward(Q, K, V, m=m, k=k, s=s, I_override=full["I"], E_override=full["E"], threads=2)
    np.testing.assert_allclose(ov["O"], full["O"], rtol=0, atol=0)
    # a different, valid override changes the output exactly as a by-hand recomputation says
    I2 = full["I"].copy(); I2[:, :, 0] = (I2[:, :, 0] + 1) % N
    I2 = np.sort(I2, axis=2)
    ov2 = oracle.forward(Q, K, V, m=m, k=k, s=s, q_ids=ids, I_override=I2, E_override=full["E"][:, ids],
                         threads=2)
    tau = 1 / math.sqrt(d)
    for h in range(2):
        for t, q in enumerate(ids):
            keys = [full["Qt"][h]] + [K[h][I2[h, e]] for e in full["E"][h, q]]
            vals = [full["Vt"][h]] + [V[h][I2[h, e]] for e in full["E"][h, q]]
            lg = tau * np.concatenate(keys) @ Q[h, q]
            w = np.exp(lg - lg.max())
            np.testing.assert_allclose(ov2["O"][h, t], w @ np.concatenate(vals) / w.sum(), rtol=1e-12)


def test_rejects_bad_parameters():
    Q = np.zeros((1, 8, 2))
    with pytest.raises(ValueError):
        oracle.forward(Q, Q, Q, m=9, k=1, s=1)
    with pytest.raises(ValueError):
        oracle.forward(Q, Q, Q, m=2, k=9, s=1)
    with pytest.raises(ValueError):
        oracle.forward(Q, Q, Q, m=2, k=1, s=3)


# ------------------------------------------------------- causal variant
# The pages describe no causal form; this build's reading (1-D pooling):
# Vt_i over the keys of landmark i's prefix (j < hi_i), a shared slot only once
# the landmark's bin is complete (hi_i <= t + 1), routed keys up to the query's
# position (j <= t), zero output when a query has no slot.

def _bins_hi(N, m):
    return np.array([-(-(i + 1) * N // m) for i in range(m)])  # ceil((i + 1) N / m)


@pytest.mark.parametrize("scale", [0.0, 0.3])
def test_causal_no_shared_full_k_is_causal_softmax_attention(scale):
    N, d, m = 96, 8, 6
    Q, K, V = (_rand((2, N, d), 40 + i) for i in range(3))
    r = oracle.forward(Q, K, V, m=m, k=N, s=1, scale=scale, no_shared=True, causal=True, threads=2)
    t = lambda a: torch.from_numpy(a)
    ref = torch.nn.functional.scaled_dot_product_attention(t(Q), t(K), t(V), is_causal=True,
                                                           scale=scale if scale > 0 else None).numpy()
    np.testing.assert_allclose(r["O"], ref, rtol=1e-12, atol=1e-12)


def test_causal_shared_full_k_is_masked_attention_over_landmarks_and_keys():
    # every key in every expert (k = N, s = 1): query t attends to the landmarks
    # of complete bins (values: attention of the landmark over its prefix) and
    # to the keys up to t, in one softmax; built here from library pooling and
    # masked SDPA
    N, d, m = 64, 5, 8
    Q, K, V = (_rand((1, N, d), 50 + i) for i in range(3))
    r = oracle.forward(Q, K, V, m=m, k=N, s=1, causal=True, threads=1)
    tq, tk, tv = (torch.from_numpy(a[0]) for a in (Q, K, V))
    Qt = torch.nn.functional.adaptive_avg_pool1d(tq.T[None], m)[0].T
    hi = _bins_hi(N, m)
    key_mask = torch.arange(N)[None, :] < torch.from_numpy(hi)[:, None]        # [m, N]: j < hi_i
    Vt = torch.nn.functional.scaled_dot_product_attention(Qt[None], tk[None], tv[None], attn_mask=key_mask[None])[0]
    np.testing.assert_allclose(r["Vt"][0], Vt.numpy(), rtol=1e-12, atol=1e-12)
    keys = torch.cat([Qt, tk])
    vals = torch.cat([Vt, tv])
    pos = torch.arange(N)[:, None]
    mask = torch.cat([torch.from_numpy(hi)[None, :] <= pos + 1, torch.arange(N)[None, :] <= pos], dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(tq[None], keys[None], vals[None], attn_mask=mask[None])[0]
    np.testing.assert_allclose(r["O"][0], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_causal_output_ignores_later_positions():
    # with every key in every expert, routes do not matter, and the output at t
    # depends on positions <= t only: changing the later ones leaves it alone
    N, d, m = 80, 4, 5
    Q, K, V = (_rand((1, N, d), 60 + i) for i in range(3))
    base = oracle.forward(Q, K, V, m=m, k=N, s=2, causal=True, threads=1)["O"][0]
    for t in (0, 15, 16, 47, 79):
        Q2, K2, V2 = Q.copy(), K.copy(), V.copy()
        rng = np.random.default_rng(t)
        for a in (Q2, K2, V2):
            a[0, t + 1:] = rng.standard_normal(a[0, t + 1:].shape)
        got = oracle.forward(Q2, K2, V2, m=m, k=N, s=2, causal=True, threads=1)["O"][0]
        np.testing.assert_allclose(got[:t + 1], base[:t + 1], rtol=1e-13, atol=1e-13)


def test_causal_query_without_slots_is_zero():
    # N = 8, m = 2 (bins [0, 4), [4, 8)), k = s = 1: key 7 is every landmark's
    # top key. Query 0 has no complete bin and its only routed key is later:
    # no slot, zero output. Query 3 completes bin 0: its only slot is
    # landmark 0, so its output is Vt_0 (attention of qt_0 over keys 0..3).
    N, d = 8, 2
    K = np.zeros((1, N, d)); K[0, 7] = [5.0, 5.0]
    Q = np.ones((1, N, d))
    V = _rand((1, N, d), 70)
    r = oracle.forward(Q, K, V, m=2, k=1, s=1, causal=True, threads=1)
    assert np.array_equal(r["I"][0], [[7], [7]])
    np.testing.assert_array_equal(r["O"][0, 0], np.zeros(d))
    np.testing.assert_allclose(r["Vt"][0, 0], V[0, :4].mean(axis=0), rtol=1e-14)  # equal scores: plain mean
    np.testing.assert_allclose(r["O"][0, 3], r["Vt"][0, 0], rtol=1e-14)


def test_causal_last_landmark_and_sets_match_noncausal():
    # the last bin ends at N, so its prefix is every key; sets and routes are
    # selected as in the non-causal pass
    N, d, m = 120, 6, 4
    Q, K, V = (_rand((1, N, d), 80 + i) for i in range(3))
    a = oracle.forward(Q, K, V, m=m, k=17, s=2, threads=1)
    b = oracle.forward(Q, K, V, m=m, k=17, s=2, causal=True, threads=1)
    np.testing.assert_array_equal(a["I"], b["I"])
    np.testing.assert_array_equal(a["E"], b["E"])
    np.testing.assert_allclose(b["Vt"][0, m - 1], a["Vt"][0, m - 1], rtol=1e-14)
    assert not np.allclose(b["Vt"][0, 0], a["Vt"][0, 0])


def test_causal_rejects_2d_pooling():
    Q = _rand((1, 64, 2), 90)
    with pytest.raises(ValueError):
        oracle.forward(Q, Q, Q, m=4, k=8, s=1, grid=(8, 8), lm=(2, 2), causal=True)


# ------------------------------------------------------------- backward
# The pages print no backward pass; oracle/backward.py is the chain rule with
# the expert sets and routes held fixed. It is pinned against central finite
# differences of the C forward oracle (run with the same sets and routes as
# overrides) and, in the special case that reduces to softmax attention,
# against PyTorch's autograd through scaled_dot_product_attention.

from oracle import backward as obwd


def _loss_fd(Q, K, V, dO, m, k, s, I, E, dirs, h=1e-5, no_shared=False):
    """Central difference of L = sum(O * dO) along the direction dirs."""
    def L(a):
        Qp, Kp, Vp = (x + a * dx for x, dx in zip((Q, K, V), dirs))
        O = oracle.forward(Qp, Kp, Vp, m, k, s, I_override=I, E_override=E, threads=1, no_shared=no_shared)["O"]
        return float(np.sum(O * dO))
    return (L(h) - L(-h)) / (2 * h)


@pytest.mark.parametrize("N,d,m,k,s,no_shared", [(48, 6, 4, 7, 2, False), (40, 5, 5, 40, 1, False),
                                                  (36, 4, 3, 9, 3, True), (30, 3, 7, 5, 2, False)])
def test_backward_matches_finite_differences(N, d, m, k, s, no_shared):
    rng = np.random.default_rng(100 + N)
    Q, K, V, dO = (rng.standard_normal((1, N, d)) for _ in range(4))
    r = oracle.forward(Q, K, V, m, k, s, threads=1, no_shared=no_shared)
    dQ, dK, dV = obwd.backward(Q, K, V, dO, r["I"], r["E"], no_shared=no_shared)
    for trial in range(3):
        dirs = [rng.standard_normal((1, N, d)) for _ in range(3)]
        fd = _loss_fd(Q, K, V, dO, m, k, s, r["I"], r["E"], dirs, no_shared=no_shared)
        an = float(np.sum(dQ * dirs[0]) + np.sum(dK * dirs[1]) + np.sum(dV * dirs[2]))
        assert abs(fd - an) <= 1e-7 * (1 + abs(fd)), (trial, fd, an)


def test_backward_each_input_alone():
    # the same check with one input perturbed at a time, so that a slip in one
    # of dQ, dK, dV cannot hide behind the others
    rng = np.random.default_rng(7)
    N, d, m, k, s = 32, 4, 4, 6, 2
    Q, K, V, dO = (rng.standard_normal((1, N, d)) for _ in range(4))
    r = oracle.forward(Q, K, V, m, k, s, threads=1)
    grads = obwd.backward(Q, K, V, dO, r["I"], r["E"])
    for which in range(3):
        dirs = [np.zeros((1, N, d)) for _ in range(3)]
        dirs[which] = rng.standard_normal((1, N, d))
        fd = _loss_fd(Q, K, V, dO, m, k, s, r["I"], r["E"], dirs)
        an = float(np.sum(grads[which] * dirs[which]))
        assert abs(fd - an) <= 1e-7 * (1 + abs(fd)), (which, fd, an)


def test_backward_no_shared_full_k_is_attention_backward():
    # shared slots off, k = N, s = 1: softmax attention, whose gradient
    # PyTorch's autograd gives through scaled_dot_product_attention
    rng = np.random.default_rng(8)
    N, d = 24, 5
    Q, K, V, dO = (rng.standard_normal((1, N, d)) for _ in range(4))
    r = oracle.forward(Q, K, V, 3, N, 1, threads=1, no_shared=True)
    dQ, dK, dV = obwd.backward(Q, K, V, dO, r["I"], r["E"], no_shared=True)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (Q, K, V))
    torch.nn.functional.scaled_dot_product_attention(tq, tk, tv).backward(torch.from_numpy(dO))
    for got, ref in ((dQ, tq.grad), (dK, tk.grad), (dV, tv.grad)):
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-10, atol=1e-12)
