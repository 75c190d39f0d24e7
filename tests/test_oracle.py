"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin comes from the pages or from mathematics: exact rational arithmetic on
tiny inputs with the fp32 error bound, closed forms, special cases that reduce
to a library routine (torch's bf16 conversion, torch's SGD with Nesterov
momentum), and invariants the method fixes. Sources:
  * "DiffuRefill-1B" model card, "How it is trained" (plain mean folded into a
    running fp32 sum as checkpoints arrive; EMA of the globals, beta 0.9);
  * "DiffuRefill-1B: Pretraining a Masked Diffusion Language Model on Free,
    Preemptible Notebook GPUs", section 3, Table 2 (plain replacement: outer
    learning rate 1, no momentum);
  * "Pythia-14M on four rented GPUs and a bucket", "Getting updates through the
    bucket" (token-weighted mean of the deltas, outer Nesterov lr 0.7 / 0.9,
    fragments and quorum), "What might explain the loss difference" (outer
    lr 1 without momentum is plain parameter averaging).
"""
import math
from fractions import Fraction as Fr

import numpy as np
import pytest
import torch

import oracle

U = Fr(1, 2 ** 24)  # unit roundoff of binary32


def ex(v) -> Fr:
    """Exact rational value of a float (fp32 values convert exactly)."""
    return Fr(float(v))


def f32(v) -> np.float32:
    return np.float32(v)


def ulps_apart(a, b) -> int:
    a = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    b = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    a = np.where(a < 0, -(a & 0x7FFFFFFF), a)
    b = np.where(b < 0, -(b & 0x7FFFFFFF), b)
    return int(np.max(np.abs(a - b))) if a.size else 0


def rng(seed=0):
    return np.random.default_rng(seed)


# ---- step a2: bf16 widening ------------------------------------------------

def test_bf16_widening_matches_torch_on_every_bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle.widen_bf16(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert (ours[~nan].view(np.uint32) == ref[~nan].view(np.uint32)).all()


def test_bf16_widening_known_values():
    bits = np.array([0x3F80, 0xC000, 0x4049, 0x0000, 0x8000, 0x7F80, 0x0001],
                    dtype=np.uint16)
    got = oracle.widen_bf16(bits)
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 3.140625
    assert got[3] == 0.0 and math.copysign(1, got[4]) == -1.0
    assert math.isinf(got[5]) and got[5] > 0
    assert got[6] == 2.0 ** -133  # smallest bf16 subnormal


# ---- steps a3/a4, plain mean ----------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_k1_replacement_returns_input_bitwise(dtype):
    r = rng(1)
    x = r.normal(0, 0.02, 4099).astype(np.float32)
    if dtype == "bf16":
        x = (x.view(np.uint32) >> 16).astype(np.uint16)
        want = oracle.widen_bf16(x)
    else:
        want = x
    theta = r.normal(0, 0.02, x.size).astype(np.float32)
    oracle.merge_tensor([x], theta, mode=oracle.MEAN_REPLACE)
    assert (theta.view(np.uint32) == want.view(np.uint32)).all()


@pytest.mark.parametrize("K", [1, 2])
def test_identical_checkpoints_average_to_themselves_bitwise(K):
    x = rng(2).normal(0, 0.02, 10007).astype(np.float32)
    got = oracle.plain_mean([x] * K)
    assert (got.view(np.uint32) == x.view(np.uint32)).all()


@pytest.mark.parametrize("K", [3, 4, 5, 8])
def test_identical_checkpoints_average_within_k_ulp(K):
    x = rng(3).normal(0, 0.02, 10007).astype(np.float32)
    got = oracle.plain_mean([x] * K)
    assert ulps_apart(got, x) <= K - 1


def test_running_sum_is_fp32_in_arrival_order():
    # 1 + 1e8 rounds to 1e8 in fp32, so arrival order (1, 1e8, -1e8) sums to 0,
    # while the exact mean is 1/3 and the order (1e8, -1e8, 1) gives fl(1/3).
    a = [np.array([v], np.float32) for v in (1.0, 1e8, -1e8)]
    assert oracle.plain_mean(a)[0] == 0.0
    b = [np.array([v], np.float32) for v in (1e8, -1e8, 1.0)]
    assert oracle.plain_mean(b)[0] == np.float32(1.0) / np.float32(3.0)


@pytest.mark.parametrize("seed", range(12))
def test_plain_mean_brute_force_exact_rational(seed):
    r = rng(100 + seed)
    K = int(r.integers(1, 9))
    scale = 10.0 ** r.integers(-6, 4)
    xs = [(r.normal(0, 1, 8) * scale).astype(np.float32) for _ in range(K)]
    got = oracle.plain_mean(xs)
    for i in range(8):
        terms = [ex(x[i]) for x in xs]
        exact = sum(terms) / K
        bound = (K + 1) * U * sum(abs(t) for t in terms) / K * Fr(101, 100)
        assert abs(ex(got[i]) - exact) <= bound


# ---- steps a3/a4, token-weighted mean of deltas ----------------------------

@pytest.mark.parametrize("seed", range(12))
def test_weighted_delta_brute_force_exact_rational(seed):
    r = rng(200 + seed)
    K = int(r.integers(1, 9))
    theta = r.normal(0, 0.02, 8).astype(np.float32)
    xs = [(theta + r.normal(0, 1e-3, 8)).astype(np.float32) for _ in range(K)]
    tokens = [int(t) for t in r.integers(200_000, 600_001, K)]
    got = oracle.weighted_delta(xs, tokens, theta)
    W = sum(tokens)
    for i in range(8):
        d = [ex(x[i]) - ex(theta[i]) for x in xs]
        exact = sum(Fr(w) * di for w, di in zip(tokens, d)) / W
        # sum is accumulated in fp32: W and every w_k must round, then K
        # subtractions, K products, K-1 additions and one division round.
        bound = (K + 4) * U * sum(Fr(w) * abs(di) for w, di in zip(tokens, d)) / W
        bound = bound * Fr(101, 100) + 4 * U * abs(exact)
        assert abs(ex(got[i]) - exact) <= bound


def test_weighted_delta_exact_on_representable_inputs():
    # Small integers, power-of-two total weight: every fp32 step is exact, so the
    # result equals sum_k w_k (x_k - theta) / W exactly. Swapped weights, a sign
    # error or a dropped worker changes it.
    theta = np.array([0, 1, -3, 10, 5, 2, 7, -1], np.float32)
    xs = [np.array([1, 2, 3, 4, 5, 6, 7, 8], np.float32),
          np.array([-2, 0, 1, 12, 5, 1, 8, 0], np.float32),
          np.array([4, 4, 4, 4, 4, 4, 4, 4], np.float32)]
    tokens = [1, 3, 4]  # W = 8
    got = oracle.weighted_delta(xs, tokens, theta)
    for i in range(8):
        exact = sum(Fr(w) * (ex(x[i]) - ex(theta[i])) for w, x in zip(tokens, xs)) / 8
        assert ex(got[i]) == exact


def test_lr1_mu0_is_token_weighted_mean_of_workers():
    r = rng(5)
    n, K = 4096, 4
    theta = r.normal(0, 0.02, n).astype(np.float32)
    xs = [(theta + r.normal(0, 1e-3, n)).astype(np.float32) for _ in range(K)]
    tokens = [250_000, 410_000, 330_001, 599_999]
    m = np.zeros(n, np.float32)
    th = theta.copy()
    oracle.merge_tensor(xs, th, mode=oracle.DELTA_NESTEROV, tokens=tokens, lr=1.0,
                        mu=0.0, m=m)
    W = sum(tokens)
    for i in range(0, n, 97):
        exact = sum(Fr(w) * ex(x[i]) for w, x in zip(tokens, xs)) / W
        delta_mag = sum(Fr(w) * abs(ex(x[i]) - ex(theta[i])) for w, x in zip(tokens, xs)) / W
        bound = 3 * U * abs(ex(theta[i])) + (K + 6) * U * delta_mag + 2 * U * abs(exact)
        assert abs(ex(th[i]) - exact) <= bound


def test_lr1_mu0_delta_equals_plain_mean_for_equal_tokens_on_exact_inputs():
    # The follow-up run of the Pythia page: outer lr 1, no momentum is averaging
    # parameters. With equal weights and exactly representable values both
    # modes give the same global.
    theta = np.array([0.5, -1.0, 2.0, 0.0], np.float32)
    xs = [np.array([1.0, 1.0, 2.0, 4.0], np.float32),
          np.array([0.0, -3.0, 2.0, -4.0], np.float32)]
    th1, m = theta.copy(), np.zeros(4, np.float32)
    oracle.merge_tensor(xs, th1, mode=oracle.DELTA_NESTEROV, tokens=[7, 7],
                        lr=1.0, mu=0.0, m=m)
    th2 = theta.copy()
    oracle.merge_tensor(xs, th2, mode=oracle.MEAN_REPLACE)
    assert (th1 == th2).all()


# ---- step a5, outer Nesterov ----------------------------------------------

def test_mu0_step_is_theta_plus_lr_delta():
    r = rng(6)
    n = 2048
    theta = r.normal(0, 1, n).astype(np.float32)
    delta = r.normal(0, 1, n).astype(np.float32)
    th, m = theta.copy(), np.zeros(n, np.float32)
    oracle.outer_nesterov(delta, 0.7, 0.0, th, m)
    lr = ex(np.float32(0.7))
    for i in range(n):
        exact = ex(theta[i]) + lr * ex(delta[i])  # theta - lr * g, g = -delta
        bound = U * abs(lr * ex(delta[i])) + U * abs(exact) + U * U * 4
        assert abs(ex(th[i]) - exact) <= bound * Fr(101, 100)
        assert m[i] == -delta[i]  # momentum 0: buffer holds g exactly


def test_nesterov_trajectory_matches_torch_sgd_nesterov():
    r = rng(7)
    n, rounds = 1000, 6
    lr, mu = 0.7, 0.9
    theta = r.normal(0, 1, n).astype(np.float32)
    deltas = [r.normal(0, 1, n).astype(np.float32) for _ in range(rounds)]
    th, m = theta.copy(), np.zeros(n, np.float32)
    p = torch.nn.Parameter(torch.from_numpy(theta.astype(np.float64)))
    opt = torch.optim.SGD([p], lr=float(np.float32(lr)), momentum=float(np.float32(mu)),
                          dampening=0.0, nesterov=True, foreach=False)
    scale = np.abs(theta.astype(np.float64))
    for d in deltas:
        oracle.outer_nesterov(d, lr, mu, th, m)
        p.grad = torch.from_numpy(-d.astype(np.float64))  # pseudo-gradient
        opt.step()
        scale = scale + 20 * np.abs(d.astype(np.float64))
    ref = p.detach().numpy()
    buf = opt.state[p]["momentum_buffer"].numpy()
    assert np.all(np.abs(th - ref) <= 1e-6 * scale)
    assert np.allclose(m, buf, rtol=1e-5, atol=1e-5)


def test_nesterov_differs_from_heavy_ball_detectably():
    # Guard for the pin above: classical momentum gives a different trajectory
    # at this tolerance, so the torch comparison does discriminate the form.
    r = rng(8)
    theta = r.normal(0, 1, 500)
    deltas = [r.normal(0, 1, 500) for _ in range(3)]
    p1 = torch.nn.Parameter(torch.tensor(theta))
    p2 = torch.nn.Parameter(torch.tensor(theta))
    o1 = torch.optim.SGD([p1], lr=0.7, momentum=0.9, nesterov=True)
    o2 = torch.optim.SGD([p2], lr=0.7, momentum=0.9, nesterov=False)
    for d in deltas:
        for p, o in ((p1, o1), (p2, o2)):
            p.grad = torch.tensor(-d)
            o.step()
    assert (p1 - p2).abs().max().item() > 0.1


# ---- step a6, EMA ------------------------------------------------------------

def test_ema_of_constant_one_is_one_minus_beta_pow_n():
    beta = np.float32(0.9)
    e = np.zeros(1, np.float32)
    one = np.ones(1, np.float32)
    b = ex(beta)
    for n in range(1, 41):
        oracle.ema(one, float(beta), e)
        exact = 1 - b ** n
        assert ulps_apart(e, np.float32(float(exact))) <= n
    # ten rounds: 1 - 0.9**10 = 0.6513215599 in exact arithmetic with beta = 0.9
    e10 = np.zeros(1, np.float32)
    for _ in range(10):
        oracle.ema(one, 0.9, e10)
    assert abs(float(e10[0]) - (1 - 0.9 ** 10)) < 5e-7


def test_ema_general_sequence_closed_form():
    r = rng(9)
    beta = np.float32(0.9)
    b, omb = ex(beta), 1 - ex(beta)  # 1 - beta is exact in fp32 (Sterbenz)
    n_el, rounds = 64, 12
    e0 = r.normal(0, 0.02, n_el).astype(np.float32)
    thetas = [r.normal(0, 0.02, n_el).astype(np.float32) for _ in range(rounds)]
    e = e0.copy()
    for t in thetas:
        oracle.ema(t, float(beta), e)
    for i in range(n_el):
        exact = b ** rounds * ex(e0[i]) + omb * sum(
            b ** (rounds - 1 - j) * ex(thetas[j][i]) for j in range(rounds))
        mag = abs(ex(e0[i])) + sum(abs(ex(t[i])) for t in thetas)
        assert abs(ex(e[i]) - exact) <= 3 * rounds * U * mag


def test_ema_weights_old_value_by_beta():
    e = np.array([1.0], np.float32)
    oracle.ema(np.array([0.0], np.float32), 0.9, e)
    assert e[0] == np.float32(0.9)


# ---- composition and drift ---------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_merge_tensor_composes_the_steps_bitwise_delta(dtype):
    r = rng(10)
    n, K = 3001, 3
    theta = r.normal(0, 0.02, n).astype(np.float32)
    xs = [(theta + r.normal(0, 1e-3, n)).astype(np.float32) for _ in range(K)]
    if dtype == "bf16":
        xs = [(x.view(np.uint32) >> 16).astype(np.uint16) for x in xs]
    tokens = [123_456, 400_000, 277_777]
    m0 = r.normal(0, 1e-3, n).astype(np.float32)
    e0 = r.normal(0, 0.02, n).astype(np.float32)
    th, m, e = theta.copy(), m0.copy(), e0.copy()
    sumsq = oracle.merge_tensor(xs, th, mode=oracle.DELTA_NESTEROV, tokens=tokens,
                                lr=0.7, mu=0.9, m=m, e=e, beta=0.9)
    d = oracle.weighted_delta(xs, tokens, theta)
    th2, m2, e2 = theta.copy(), m0.copy(), e0.copy()
    oracle.outer_nesterov(d, 0.7, 0.9, th2, m2)
    oracle.ema(th2, 0.9, e2)
    assert (th.view(np.uint32) == th2.view(np.uint32)).all()
    assert (m.view(np.uint32) == m2.view(np.uint32)).all()
    assert (e.view(np.uint32) == e2.view(np.uint32)).all()
    assert sumsq == pytest.approx(math.fsum(float(v) ** 2 for v in d), rel=1e-12)


def test_merge_tensor_composes_the_steps_bitwise_mean():
    r = rng(11)
    n, K = 2049, 5
    theta = r.normal(0, 0.02, n).astype(np.float32)
    xs = [(theta + r.normal(0, 2e-3, n)).astype(np.float32) for _ in range(K)]
    e0 = theta.copy()
    th, e = theta.copy(), e0.copy()
    sumsq = oracle.merge_tensor(xs, th, mode=oracle.MEAN_REPLACE, e=e, beta=0.9)
    mean = oracle.plain_mean(xs)
    e2 = e0.copy()
    oracle.ema(mean, 0.9, e2)
    assert (th.view(np.uint32) == mean.view(np.uint32)).all()
    assert (e.view(np.uint32) == e2.view(np.uint32)).all()
    drift = (mean - theta).astype(np.float32)
    assert sumsq == pytest.approx(math.fsum(float(v) ** 2 for v in drift), rel=1e-12)


def test_drift_sum_of_squares_exact_small():
    theta = np.array([0.0, 0.0, 0.0], np.float32)
    xs = [np.array([3.0, 4.0, 0.0], np.float32)]
    assert oracle.merge_tensor(xs, theta.copy(), mode=oracle.MEAN_REPLACE) == 25.0


def test_rejects_bad_arguments():
    x = np.zeros(4, np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.weighted_delta([x], [0], x)           # total weight zero
    with pytest.raises(oracle.OracleError):
        oracle.weighted_delta([x], [-1, 2][:1], x)   # negative weight
    with pytest.raises(oracle.OracleError):
        oracle.merge_tensor([x], x.copy(), mode=oracle.DELTA_NESTEROV, tokens=[1])


# ---- round level: fragments, quorum, stale rounds ----------------------------

def _round_state(n_tensors=6, n=33, frags=(0, 0, 1, 1, 2, 3), seed=12):
    r = rng(seed)
    theta = [r.normal(0, 0.02, n).astype(np.float32) for _ in range(n_tensors)]
    st = oracle.OracleState(theta=[t.copy() for t in theta],
                            m=[np.zeros(n, np.float32) for _ in range(n_tensors)],
                            e=[t.copy() for t in theta], fragment_of=list(frags))
    ck = [[(t + r.normal(0, 1e-3, n)).astype(np.float32) for t in theta] for _ in range(4)]
    return st, ck


def test_round_touches_only_its_fragment_and_included_workers():
    st, ck = _round_state()
    before = [t.copy() for t in st.theta]
    ck[2] = [np.full_like(t, np.nan) for t in ck[2]]  # masked worker: never read
    norms, frag = oracle.merge_round(st, round=0, fragment=1, ckpts=ck,
                                     included=[3, 0, 1], tokens=[5, 6, 7, 8],
                                     mode=oracle.DELTA_NESTEROV, lr=0.7, mu=0.9,
                                     quorum=3, ema_beta=0.9)
    for t in range(6):
        if st.fragment_of[t] == 1:
            assert np.isfinite(st.theta[t]).all() and not (st.theta[t] == before[t]).all()
        else:
            assert (st.theta[t].view(np.uint32) == before[t].view(np.uint32)).all()
            assert (st.m[t] == 0).all()
    assert len(norms) == 2 and frag == pytest.approx(math.sqrt(sum(v * v for v in norms)))


def test_quorum_and_stale_round_rejected():
    st, ck = _round_state()
    with pytest.raises(oracle.QuorumError):
        oracle.merge_round(st, round=0, fragment=0, ckpts=ck, included=[0, 1],
                           tokens=[1] * 4, mode=oracle.DELTA_NESTEROV, quorum=3)
    oracle.merge_round(st, round=5, fragment=0, ckpts=ck, included=[0, 1, 2],
                       tokens=[1] * 4, mode=oracle.DELTA_NESTEROV, quorum=3)
    with pytest.raises(oracle.StaleRoundError):
        oracle.merge_round(st, round=5, fragment=1, ckpts=ck, included=[0, 1, 2],
                           tokens=[1] * 4, mode=oracle.DELTA_NESTEROV, quorum=3)


def test_rounds_on_disjoint_fragments_commute():
    a, ck = _round_state(seed=13)
    b, _ = _round_state(seed=13)
    kw = dict(ckpts=ck, included=[0, 2, 3], tokens=[9, 8, 7, 6],
              mode=oracle.DELTA_NESTEROV, lr=0.7, mu=0.9, quorum=3, ema_beta=0.9)
    oracle.merge_round(a, round=0, fragment=0, **kw)
    oracle.merge_round(a, round=1, fragment=3, **kw)
    oracle.merge_round(b, round=0, fragment=3, **kw)
    oracle.merge_round(b, round=1, fragment=0, **kw)
    for t in range(6):
        assert (a.theta[t].view(np.uint32) == b.theta[t].view(np.uint32)).all()
        assert (a.e[t].view(np.uint32) == b.e[t].view(np.uint32)).all()


def test_fragment_minus_one_is_all_tensors():
    assert oracle.fragment_tensors([0, 1, 2, 1], -1) == [0, 1, 2, 3]
    assert oracle.fragment_tensors([0, 1, 2, 1], 1) == [1, 3]
    assert oracle.fragment_tensors([0, 1, 2, 1], 4) == []


# ---- uniform average of the globals (SWA) and snapshot averages -------------------

def test_swa_first_global_is_copied_exactly():
    theta = rng(20).normal(0, 0.02, 1001).astype(np.float32)
    mu = np.zeros(1001, np.float32)
    oracle.swa(theta, 1, mu)
    assert bitwise_equal_np(mu, theta)


def bitwise_equal_np(a, b):
    return (np.asarray(a, np.float32).view(np.uint32) == np.asarray(b, np.float32).view(np.uint32)).all()


def test_swa_of_a_constant_stays_exact():
    mu = np.zeros(64, np.float32)
    c = rng(21).normal(0, 0.02, 64).astype(np.float32)
    for n in range(1, 131):
        oracle.swa(c, n, mu)
        assert bitwise_equal_np(mu, c)


def test_swa_is_the_uniform_average_of_130_globals():
    # the released weights: the uniform average of the 130 globals of the
    # final stretch (technical report, section 4 and Table 5)
    r = rng(22)
    n_el, n = 48, 130
    thetas = [r.normal(0, 0.02, n_el).astype(np.float32) for _ in range(n)]
    mu = np.zeros(n_el, np.float32)
    for j, t in enumerate(thetas, 1):
        oracle.swa(t, j, mu)
    for i in range(n_el):
        exact = sum(ex(t[i]) for t in thetas) / n
        mag = max(abs(ex(t[i])) for t in thetas)
        assert abs(ex(mu[i]) - exact) <= 4 * n * U * mag


def test_swa_rejects_a_zero_count():
    with pytest.raises(oracle.OracleError):
        oracle.swa(np.zeros(4, np.float32), 0, np.zeros(4, np.float32))


def test_snapshot_average_is_their_plain_mean():
    # "average of the last 3 / 5 snapshots" (technical report, Table 5)
    r = rng(23)
    snaps = [r.normal(0, 0.02, 8).astype(np.float32) for _ in range(5)]
    for w in (3, 5):
        got = oracle.plain_average(snaps[-w:])
        for i in range(8):
            exact = sum(ex(s[i]) for s in snaps[-w:]) / w
            assert abs(ex(got[i]) - exact) <= (w + 1) * U * sum(abs(ex(s[i])) for s in snaps[-w:])


def test_round_level_swa_tracks_the_rounds_globals():
    st, ck = _round_state(seed=24)
    st.swa = [np.zeros_like(t) for t in st.theta]
    st.swa_count = [0] * len(st.theta)
    seen = {t: [] for t in range(6)}
    for rnd in range(3):
        oracle.merge_round(st, round=rnd, fragment=-1, ckpts=ck, included=[0, 1, 2],
                           tokens=[1, 2, 3, 4], mode=oracle.DELTA_NESTEROV, lr=0.7, mu=0.9,
                           quorum=3, swa_update=True)
        for t in range(6):
            seen[t].append(st.theta[t].copy())
    for t in range(6):
        assert st.swa_count[t] == 3
        exact = [sum(ex(s[i]) for s in seen[t]) / 3 for i in range(st.theta[t].size)]
        for i, x in enumerate(exact):
            assert abs(ex(st.swa[t][i]) - x) <= 12 * U * max(abs(ex(s[i])) for s in seen[t])


# ---- per-worker drift and keep-drift adoption (technical report, section 5.1) -----

def test_worker_drift_matches_fsum_and_exact_case():
    r = rng(30)
    theta = r.normal(0, 0.02, 777).astype(np.float32)
    xs = [(theta + r.normal(0, s, 777)).astype(np.float32) for s in (1e-3, 2e-3, 5e-4)]
    got = oracle.worker_drift(xs, theta)
    for x, v in zip(xs, got):
        d = (x - theta).astype(np.float32)
        assert v == pytest.approx(math.fsum(float(a) ** 2 for a in d), rel=1e-12)
    assert got[1] > got[0] > got[2]          # ordered like the noise scales
    t0 = np.zeros(2, np.float32)
    assert oracle.worker_drift([np.array([3.0, 4.0], np.float32),
                                np.array([0.0, 1.0], np.float32)], t0) == [25.0, 1.0]


def test_worker_drift_bf16_uses_widened_values():
    theta = np.zeros(2, np.float32)
    x = np.array([0x3F80, 0xC000], np.uint16)  # 1.0, -2.0
    assert oracle.worker_drift([x], theta) == [5.0]


def test_keep_drift_adoption_exact_and_bounded():
    # theta_w + (g - pushed): exact on representable inputs; a worker that did
    # not move since its push lands on the global.
    tw = np.array([1.0, 2.0, -3.0, 0.5], np.float32)
    g = np.array([4.0, -2.0, 0.0, 0.25], np.float32)
    p = np.array([0.5, 2.0, -1.0, 0.5], np.float32)
    out = tw.copy()
    oracle.adopt_keep_drift(out, g, p)
    assert list(out) == [4.5, -2.0, -2.0, 0.25]
    r = rng(31)
    pushed = r.normal(0, 0.02, 500).astype(np.float32)
    glob = (pushed + r.normal(0, 1e-3, 500)).astype(np.float32)
    same = pushed.copy()
    oracle.adopt_keep_drift(same, glob, pushed)   # no progress since the push
    for i in range(500):                           # lands on the global (two roundings)
        assert abs(ex(same[i]) - ex(glob[i])) <= 2 * U * (abs(ex(pushed[i])) + abs(ex(glob[i])))
    tw = (pushed + r.normal(0, 1e-3, 500)).astype(np.float32)
    out = tw.copy()
    oracle.adopt_keep_drift(out, glob, pushed)
    for i in range(500):
        exact = ex(tw[i]) + ex(glob[i]) - ex(pushed[i])
        bound = 2 * U * (abs(exact) + abs(ex(glob[i]) - ex(pushed[i])))
        assert abs(ex(out[i]) - exact) <= bound


def test_keep_drift_adoption_bf16_pushed():
    tw = np.array([1.0, 1.0], np.float32)
    g = np.array([2.0, 0.0], np.float32)
    pushed = np.array([0x3F80, 0xBF80], np.uint16)   # 1.0, -1.0
    oracle.adopt_keep_drift(tw, g, pushed)
    assert list(tw) == [2.0, 2.0]


# ---- outer orthogonalisation (technical report, section 5.3) ---------------------

def _orthonormal(rng_, m, r):
    q, _ = np.linalg.qr(rng_.normal(size=(m, r)))
    return q


@pytest.mark.parametrize("m,n", [(40, 12), (12, 40), (25, 25)])
def test_polar_of_a_known_svd_is_q_p_transposed(m, n):
    r_ = rng(40 + m)
    k = min(m, n)
    q, p = _orthonormal(r_, m, k), _orthonormal(r_, n, k)
    s = r_.uniform(0.1, 5.0, k)
    got = oracle.polar(q @ np.diag(s) @ p.T)
    assert np.allclose(got, q @ p.T, atol=1e-12)


@pytest.mark.parametrize("m,n", [(30, 10), (10, 30)])
def test_polar_agrees_with_the_inverse_square_root_route(m, n):
    d = rng(41).normal(size=(m, n))
    w, v = np.linalg.eigh(d.T @ d if m >= n else d @ d.T)
    inv_sqrt = v @ np.diag(w ** -0.5) @ v.T
    want = d @ inv_sqrt if m >= n else inv_sqrt @ d
    assert np.allclose(oracle.polar(d), want, atol=1e-10)


def test_polar_is_scale_invariant_and_semi_orthogonal():
    d = rng(42).normal(size=(20, 7))
    o = oracle.polar(d)
    assert np.allclose(oracle.polar(3.7 * d), o, atol=1e-12)
    assert np.allclose(o.T @ o, np.eye(7), atol=1e-12)
    assert np.allclose(oracle.polar(o), o, atol=1e-12)


@pytest.mark.parametrize("mode", [oracle.ORTHO_SCALE_FIXED, oracle.ORTHO_SCALE_MATCH_NORM])
def test_orthogonal_update_magnitude(mode):
    r_ = rng(43)
    m, n = 16, 6
    theta = r_.normal(0, 0.02, m * n).astype(np.float32)
    xs = [(theta + r_.normal(0, 1e-3, m * n)).astype(np.float32) for _ in range(3)]
    new, delta = oracle.orthogonal_update(xs, theta, m, lr=0.5, scale_mode=mode)
    step = new - theta.astype(np.float64)
    fro = math.sqrt(float(np.sum(step ** 2)))
    if mode == oracle.ORTHO_SCALE_FIXED:
        assert fro == pytest.approx(0.5 * math.sqrt(n), rel=1e-10)
    else:
        assert fro == pytest.approx(0.5 * math.sqrt(float(np.sum(delta.astype(np.float64) ** 2))),
                                    rel=1e-10)
    # the step points along the update: <step, Delta> = s * nuclear norm > 0
    assert float(np.sum(step * delta.astype(np.float64))) > 0
    assert np.array_equal(delta, (oracle.plain_mean(xs) - theta).astype(np.float32))
