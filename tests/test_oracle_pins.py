"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin is a function of the oracle build (``mutant``) so that the last test
can show that a planted mistake in the oracle fails at least one pin.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import chunkwise_naive, rel_err, unrolled_bruteforce

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(T, dk, dv, seed, g_scale=5.0, s0_std=0.5):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((T, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.standard_normal((T, dk))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    v = rng.standard_normal((T, dv))
    g = -g_scale / (1.0 + np.exp(-rng.standard_normal((T, dk))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    S0 = s0_std * rng.standard_normal((dk, dv))
    f32 = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    return f32(q), f32(k), f32(v), f32(g), f32(beta), f32(S0)


def _run1(q, k, v, g, beta, S0, mutant=0):
    """Oracle on one (sequence, head)."""
    T = q.shape[0]
    o, f = oracle.recurrent(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None],
                            np.array([0, T], dtype=np.int32), None if S0 is None else S0[None, None],
                            threads=1, mutant=mutant)
    return o[:, 0], f[0, 0]


# ---------------------------------------------------------------- pins
def pin_delta_invariant(mutant=0, dk=16, dv=16):
    """g = 0, beta = 1, orthonormal keys: the state returns each written value exactly
    (Q05: the write subtracts the old prediction).  Returns the max error."""
    n = dk
    K = oracle.delta_invariant_keys(dk, n, seed=3).astype(np.float32)
    rng = np.random.default_rng(4)
    V = rng.standard_normal((n, dv)).astype(np.float32)
    S0 = (0.3 * rng.standard_normal((dk, dv))).astype(np.float32)
    g = np.zeros((n, dk), np.float32)
    beta = np.ones(n, np.float32)
    _, S = _run1(K, K, V, g, beta, S0, mutant)
    # keys are the fp32-rounded QR rows; the invariant holds for exactly orthonormal
    # keys, so compare against the prediction for the keys actually stored
    Kd = K.astype(np.float64)
    Vd = V.astype(np.float64)
    G = Kd @ Kd.T
    assert np.max(np.abs(G - np.eye(n))) < 1e-6
    return float(np.max(np.abs(S.T @ Kd.T - Vd.T)))


def pin_repeated_key_overwrites(mutant=0):
    """Lab A toy (hand-worked): a repeated key returns its latest value, not a sum."""
    with open(os.path.join(GOLDEN, "lab_a_delta_toy.json")) as fh:
        fx = json.load(fh)
    f32 = lambda a: np.asarray(a, dtype=np.float32)
    o, S = _run1(f32(fx["q"]), f32(fx["k"]), f32(fx["v"]), f32(fx["g"]), f32(fx["beta"]), None, mutant)
    return max(float(np.max(np.abs(o - np.asarray(fx["expected_out"])))),
               float(np.max(np.abs(S - np.asarray(fx["expected_final_state"])))))


def pin_bruteforce(mutant=0, dk=6, dv=6, T=8, seed=11):
    """Explicit product of transition matrices, T <= 8."""
    q, k, v, g, beta, S0 = _rand_case(T, dk, dv, seed)
    o, S = _run1(q, k, v, g, beta, S0, mutant)
    ou, Su = unrolled_bruteforce(q, k, v, g, beta, S0)
    return max(rel_err(o, ou), rel_err(S, Su))


def pin_chunkwise(mutant=0, dk=8, dv=8, T=70, C=16, seed=5):
    """Naive chunkwise rewrite (explicit inverse) equals the recurrence."""
    q, k, v, g, beta, S0 = _rand_case(T, dk, dv, seed)
    o, S = _run1(q, k, v, g, beta, S0, mutant)
    oc, Sc = chunkwise_naive(q, k, v, g, beta, S0, chunk=C)
    return max(rel_err(o, oc), rel_err(S, Sc))


def pin_closed_form_no_write(mutant=0, dk=8, dv=5, T=9, seed=6):
    """beta = 0: S_t = Diag(exp sum g) S_0 and o_t = S_t^T q_t."""
    q, k, v, g, beta, S0 = _rand_case(T, dk, dv, seed, g_scale=1.0)
    beta[:] = 0
    o, S = _run1(q, k, v, g, beta, S0, mutant)
    G = np.cumsum(g.astype(np.float64), axis=0)
    ref_o = np.stack([(np.exp(G[t])[:, None] * S0).T @ q[t] for t in range(T)])
    ref_S = np.exp(G[-1])[:, None] * S0
    return max(rel_err(o, ref_o), rel_err(S, ref_S))


def pin_closed_form_first_token(mutant=0, dk=8, dv=5, seed=7):
    """S_0 = 0: o_1 = beta_1 (k_1 . q_1) v_1 whatever g_1 is."""
    q, k, v, g, beta, _ = _rand_case(1, dk, dv, seed)
    o, _ = _run1(q, k, v, g, beta, None, mutant)
    ref = float(beta[0]) * float(np.dot(k[0].astype(np.float64), q[0])) * v[0].astype(np.float64)
    return rel_err(o[0], ref)


# ---------------------------------------------------------------- tests on the real oracle
def test_delta_rule_invariant():
    assert pin_delta_invariant() < 1e-6
    assert pin_delta_invariant(dk=32, dv=8) < 1e-6


def test_repeated_key_overwrites_lab_a():
    assert pin_repeated_key_overwrites() < 1e-12
    # and the additive alternative the lab contrasts is really different
    with open(os.path.join(GOLDEN, "lab_a_delta_toy.json")) as fh:
        fx = json.load(fh)
    assert fx["additive_final_state"] != fx["expected_final_state"]


@pytest.mark.parametrize("dk,dv,T", [(6, 6, 8), (5, 3, 7), (3, 7, 8), (4, 4, 1)])
def test_bruteforce_unrolling(dk, dv, T):
    assert pin_bruteforce(dk=dk, dv=dv, T=T) < 1e-12


@pytest.mark.parametrize("C", [1, 3, 16, 64])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 150])
def test_chunkwise_rewrite(C, T):
    assert pin_chunkwise(T=T, C=C, dk=8, dv=6) < 1e-10


def test_chunkwise_rewrite_full_head_dim():
    assert pin_chunkwise(dk=128, dv=128, T=200, C=64, seed=9) < 1e-10


def test_closed_forms():
    assert pin_closed_form_no_write() < 1e-12
    assert pin_closed_form_first_token() < 1e-12
    # g = 0, beta = 0: o_t = S_0^T q_t
    q, k, v, g, beta, S0 = _rand_case(5, 8, 4, 8)
    g[:] = 0
    beta[:] = 0
    o, _ = _run1(q, k, v, g, beta, S0)
    assert rel_err(o, q.astype(np.float64) @ S0.astype(np.float64)) < 1e-12


def test_linear_in_values_and_initial_state():
    """For fixed q, k, g, beta the recurrence is linear in (v, S_0): the outputs and the
    final state of a*(v1, S01) + b*(v2, S02) are a*(run 1) + b*(run 2).  Inputs are
    chosen exactly representable in fp32 so that the combination is exact."""
    q, k, v1, g, beta, S01 = _rand_case(12, 8, 6, 21)
    _, _, v2, _, _, S02 = _rand_case(12, 8, 6, 22)
    dy = lambda x: (np.round(x * 64.0) / 64.0).astype(np.float32)   # dyadic: sums below stay exact
    v1, v2, S01, S02 = dy(v1), dy(v2), dy(S01), dy(S02)
    a, b = 0.5, -2.0
    o1, f1 = _run1(q, k, v1, g, beta, S01)
    o2, f2 = _run1(q, k, v2, g, beta, S02)
    o, f = _run1(q, k, (a * v1 + b * v2).astype(np.float32), g, beta, (a * S01 + b * S02).astype(np.float32))
    assert rel_err(o, a * o1 + b * o2) < 1e-12 and rel_err(f, a * f1 + b * f2) < 1e-12


def test_query_only_reads():
    """q enters only the read-out: scaling q scales every output and leaves the state
    trajectory (hence the final state) untouched; a zero q gives zero outputs."""
    q, k, v, g, beta, S0 = _rand_case(10, 8, 8, 23)
    o1, f1 = _run1(q, k, v, g, beta, S0)
    o2, f2 = _run1((4.0 * q).astype(np.float32), k, v, g, beta, S0)
    o0, f0 = _run1(np.zeros_like(q), k, v, g, beta, S0)
    assert rel_err(o2, 4.0 * o1) < 1e-12
    assert np.array_equal(f2, f1) and np.array_equal(f0, f1)
    assert np.all(o0 == 0)


def test_norm_bound():
    """||k|| = 1, beta in [0,1], g <= 0 make (I - beta k k^T) Diag(e^g) a contraction:
    ||S_t||_2 <= ||S_{t-1}||_2 + beta_t ||v_t||."""
    q, k, v, g, beta, S0 = _rand_case(40, 16, 16, 10)
    S = S0
    for t in range(40):
        _, Sn = _run1(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], beta[t:t + 1], S.astype(np.float32))
        lhs = np.linalg.norm(Sn, 2)
        rhs = np.linalg.norm(S.astype(np.float32).astype(np.float64), 2) + beta[t] * np.linalg.norm(v[t])
        assert lhs <= rhs * (1 + 1e-9)
        S = Sn


def test_varlen_equals_independent_runs_and_heads_independent():
    rng = np.random.default_rng(12)
    lens = [5, 1, 17, 9]
    T, H, dk, dv = sum(lens), 3, 8, 6
    cases = [_rand_case(T, dk, dv, 100 + h) for h in range(H)]
    st = lambda i: np.ascontiguousarray(np.stack([c[i] for c in cases], axis=1))
    q, k, v, g, beta = st(0), st(1), st(2), st(3), st(4)
    S0 = (0.1 * rng.standard_normal((len(lens), H, dk, dv))).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o, S = oracle.recurrent(q, k, v, g, beta, cu, S0, threads=4)
    for n in range(len(lens)):
        for h in range(H):
            b, e = cu[n], cu[n + 1]
            on, Sn = _run1(q[b:e, h], k[b:e, h], v[b:e, h], g[b:e, h], beta[b:e, h], S0[n, h])
            assert np.array_equal(on, o[b:e, h])
            assert np.array_equal(Sn, S[n, h])


def test_chained_calls_equal_one_shot():
    """Carrying final_state into init_state reproduces the one-shot run (up to the fp32 hand-off)."""
    q, k, v, g, beta, S0 = _rand_case(50, 8, 8, 13)
    o, S = _run1(q, k, v, g, beta, S0)
    o1, S1 = _run1(q[:20], k[:20], v[:20], g[:20], beta[:20], S0)
    o2, S2 = _run1(q[20:], k[20:], v[20:], g[20:], beta[20:], S1.astype(np.float32))
    assert rel_err(np.concatenate([o1, o2]), o) < 1e-6
    assert rel_err(S2, S) < 1e-6


def test_bf16_inputs_widen_exactly():
    import torch
    q, k, v, g, beta, S0 = _rand_case(12, 8, 8, 14)
    tb = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    qb, kb, vb = tb(q), tb(k), tb(v)
    o_b, S_b = _run1(qb, kb, vb, g, beta, S0)
    o_f, S_f = _run1(qb.float().numpy(), kb.float().numpy(), vb.float().numpy(), g, beta, S0)
    assert np.array_equal(o_b, o_f) and np.array_equal(S_b, S_f)


def test_bounded_decay_lab_b_closed_form():
    """Lab B: with log-decay bounded below by g_min = -5, the largest reciprocal of the
    cumulative decay inside an L-token tile is exp(5 (L - 1)).  L = 16 stays finite in
    fp32 and bf16 (about 3.7e32); L = 64 (exp(315)) overflows both."""
    f32_max = float(np.finfo(np.float32).max)
    bf16_max = 3.3895313892515355e38
    worst = lambda L: 5.0 * (L - 1)
    assert np.exp(worst(16)) < bf16_max and np.exp(worst(16)) < f32_max
    assert abs(np.exp(worst(16)) - 3.733241996799e32) / 3.733241996799e32 < 1e-9
    assert worst(64) > np.log(f32_max)
    # the sub-tile-relative factors used by the GPU path lie in [exp(-80), 1] and [1, exp(80)]
    assert np.exp(-80.0) > np.finfo(np.float32).tiny and np.exp(80.0) < f32_max


def test_oracle_rejects_bad_cu_seqlens():
    q, k, v, g, beta, _ = _rand_case(4, 4, 4, 1)
    with pytest.raises(ValueError):
        oracle.recurrent(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None],
                         np.array([0, 3, 2], dtype=np.int32))


# ---------------------------------------------------------------- planted mistakes
ALL_PINS = [pin_delta_invariant, pin_repeated_key_overwrites, pin_bruteforce, pin_chunkwise,
            pin_closed_form_no_write, pin_closed_form_first_token]


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5])
def test_each_planted_oracle_mistake_fails_a_pin(mutant, tmp_path):
    path = oracle.build_oracle(mutant=mutant, out_dir=str(tmp_path))
    assert oracle.kda_ref._lib(path=path).kda_oracle_mutant() == mutant
    errs = {}
    for pin in ALL_PINS:
        # route the pin through the mutant build
        saved = oracle.kda_ref._LIBS.get(mutant)
        oracle.kda_ref._LIBS[mutant] = oracle.kda_ref._lib(path=path)
        try:
            errs[pin.__name__] = pin(mutant=mutant)
        finally:
            if saved is None:
                oracle.kda_ref._LIBS.pop(mutant, None)
            else:
                oracle.kda_ref._LIBS[mutant] = saved
    assert max(errs.values()) > 1e-3, errs


# ---------------------------------------------------------------- the input prologue
def test_prologue_closed_forms():
    """The oracle's input prologue against values its definition fixes: a 3-4-5 row becomes
    (0.6, 0.8), exactly in fp32 and as the nearest bf16 values (0.6015625, 0.80078125) in
    bf16; a zero row stays zero (the 1e-12 floor); sigmoid(0) = 1/2 and sigmoid(ln 3) = 3/4
    give g = -2.5, -3.75 and beta = 0.5, 0.75; logits of +-1e4 give the limits without NaN."""
    import torch
    raw = torch.zeros(2, 1, 8)
    raw[0, 0, 0], raw[0, 0, 1] = 3.0, 4.0
    z = torch.tensor([[0.0], [float(np.log(3.0))]]).repeat(1, 4).reshape(2, 1, 4)
    y = torch.tensor([[0.0], [float(np.log(3.0))]])
    d = {"q": raw.clone(), "k": raw.clone(), "g": z, "beta": y}
    p = oracle.prologue(d, oracle.PROLOGUE_QK_L2NORM | oracle.PROLOGUE_G_LOGITS | oracle.PROLOGUE_BETA_LOGITS)
    for name in ("q", "k"):
        assert p[name].dtype == torch.float32
        assert p[name][0, 0, 0].item() == np.float32(0.6) and p[name][0, 0, 1].item() == np.float32(0.8)
        assert torch.count_nonzero(p[name][0, 0, 2:]) == 0 and torch.count_nonzero(p[name][1]) == 0
    assert np.allclose(p["g"][:, 0, 0].numpy(), [-2.5, -3.75], rtol=0, atol=1e-6)
    assert np.allclose(p["beta"][:, 0].numpy(), [0.5, 0.75], rtol=0, atol=1e-7)
    pb = oracle.prologue({"q": raw.to(torch.bfloat16), "k": raw.to(torch.bfloat16)}, oracle.PROLOGUE_QK_L2NORM)
    assert pb["q"].dtype == torch.bfloat16
    assert pb["q"][0, 0, 0].item() == 0.6015625 and pb["q"][0, 0, 1].item() == 0.80078125
    lim = oracle.prologue({"g": torch.tensor([[[1e4, -1e4]]]), "beta": torch.tensor([[1e4], [-1e4]])},
                          oracle.PROLOGUE_G_LOGITS | oracle.PROLOGUE_BETA_LOGITS)
    assert lim["g"].flatten().tolist() == [-5.0, -0.0] and lim["beta"].flatten().tolist() == [1.0, 0.0]
    # only the asked-for bits act
    only_g = oracle.prologue(d, oracle.PROLOGUE_G_LOGITS)
    assert torch.equal(only_g["q"], d["q"]) and torch.equal(only_g["beta"], d["beta"])


def test_prologue_scale_invariance_and_unit_norm():
    """Normalisation ignores a positive scale of the row, and every non-zero row comes out
    with norm 1 (to fp32 rounding)."""
    import torch
    rng = np.random.default_rng(31)
    x = torch.from_numpy(rng.standard_normal((40, 3, 64)).astype(np.float32))
    a = oracle.prologue({"q": x, "k": x}, oracle.PROLOGUE_QK_L2NORM)["q"]
    b = oracle.prologue({"q": 8.0 * x, "k": x}, oracle.PROLOGUE_QK_L2NORM)["q"]
    assert torch.equal(a, b)   # scaling by a power of two is exact
    c = oracle.prologue({"q": 3.7 * x, "k": x}, oracle.PROLOGUE_QK_L2NORM)["q"]
    assert float((a - c).abs().max()) < 1e-6
    n = torch.linalg.vector_norm(a.double(), dim=-1)
    assert float((n - 1).abs().max()) < 1e-6


def test_prologue_keeps_the_delta_invariant():
    """Raw keys = orthonormal keys times arbitrary positive scales, g logits of -1e4 (g = 0)
    and beta logits of +1e4 (beta = 1): after the prologue the keys are orthonormal again,
    so the recurrence returns each written value (the invariant of the delta rule)."""
    import torch
    dk = dv = 16
    K = oracle.delta_invariant_keys(dk, dk, seed=5)
    rng = np.random.default_rng(6)
    scales = rng.uniform(0.1, 20.0, size=(dk, 1))
    raw = torch.from_numpy((K * scales)[:, None, :].astype(np.float32))
    V = rng.standard_normal((dk, dv)).astype(np.float32)
    d = {"q": raw, "k": raw, "g": torch.full((dk, 1, dk), -1e4), "beta": torch.full((dk, 1), 1e4)}
    p = oracle.prologue(d, oracle.PROLOGUE_QK_L2NORM | oracle.PROLOGUE_G_LOGITS | oracle.PROLOGUE_BETA_LOGITS)
    assert torch.count_nonzero(p["g"]) == 0 and bool((p["beta"] == 1).all())
    Kn = p["k"][:, 0].numpy()
    _, S = _run1(Kn, Kn, V, p["g"][:, 0].numpy(), p["beta"][:, 0].numpy(), None)
    Kd = Kn.astype(np.float64)
    assert np.max(np.abs(Kd @ Kd.T - np.eye(dk))) < 1e-6
    assert np.max(np.abs(S.T @ Kd.T - V.astype(np.float64).T)) < 1e-5


def test_rel_err_hand_worked_values():
    """The parity bar's measure, max |x - ref| / RMS(ref), on values worked out by hand.
    Each case tells it apart from a plausible slip: the mean instead of the max of |x - ref|,
    the L2 norm or the standard deviation of ref instead of its RMS, the RMS over the
    non-zero entries only, or a sign taken one way."""
    ref = np.array([1.0, -1.0, 1.0, -1.0])           # RMS 1, L2 norm 2
    x = ref + np.array([0.0, 0.5, -0.25, 0.0])       # max |d| 0.5, mean |d| 0.1875
    assert rel_err(x, ref) == 0.5
    assert rel_err(ref - (x - ref), ref) == 0.5      # errors of the other sign
    ref = np.array([2.0, 2.0, 2.0, 2.0, 0.0, 0.0, 0.0, 0.0])   # RMS sqrt(2); std 1; RMS of non-zeros 2
    x = ref.copy()
    x[7] = 1.0
    assert abs(rel_err(x, ref) - 1.0 / np.sqrt(2.0)) < 1e-15
    ref2 = np.array([[3.0, 4.0, 0.0], [0.0, 0.0, 5.0]])        # RMS sqrt(50 / 6) = 5 / sqrt(3)
    x2 = ref2 + np.array([[0.0, 0.0, 0.0], [0.0, -2.5, 0.0]])
    assert abs(rel_err(x2, ref2) - 2.5 * np.sqrt(3.0) / 5.0) < 1e-15
    # an all-zero reference: the bar falls back to the absolute error
    assert rel_err(np.array([0.0, 0.25, -0.5]), np.zeros(3)) == 0.5
    assert rel_err(np.zeros(0), np.zeros(0)) == 0.0
    assert rel_err(ref2, ref2) == 0.0


def test_output_gate_closed_forms():
    """The oracle's output gate o * sigmoid(z) at points where sigmoid is known exactly:
    z = 0 halves o, z = ln 3 gives 3/4, z = +-1e4 gives o and 0, sigmoid(z) + sigmoid(-z) = 1,
    and it acts channel by channel.  Catches tanh for sigmoid, a sign flip of z, o and z
    swapped, or a reduction over the channels."""
    rng = np.random.default_rng(41)
    o = rng.standard_normal((5, 3, 16))
    z = rng.standard_normal((5, 3, 16))
    assert np.array_equal(oracle.output_gate(o, np.zeros_like(o)), 0.5 * o)
    assert np.max(np.abs(oracle.output_gate(o, np.full_like(o, np.log(3.0))) - 0.75 * o)) < 1e-15
    assert np.array_equal(oracle.output_gate(o, np.full_like(o, 1e4)), o)
    assert np.array_equal(oracle.output_gate(o, np.full_like(o, -1e4)), np.zeros_like(o))
    assert np.max(np.abs(oracle.output_gate(o, z) + oracle.output_gate(o, -z) - o)) < 1e-15
    z2 = z.copy()
    z2[2, 1, 7] += 3.0
    diff = oracle.output_gate(o, z2) != oracle.output_gate(o, z)
    assert diff.sum() == 1 and diff[2, 1, 7]


def test_range_transition_and_split_identity():
    """Context-parallel prefill rests on the recurrence being affine in its initial state: a
    token range maps the state entering it to M S + S_r.  M, the state after the range from
    S_0 = I with v = 0, equals the explicit product of the per-token transitions
    (I - beta_t k_t k_t^T) Diag(e^{g_t}) (written out here, T = 7); and splitting a sequence at
    any token, then combining, reproduces the one-shot final state and the later outputs."""
    dk = 6
    q, k, v, g, beta, _ = _rand_case(7, dk, dk, 31, g_scale=1.0)
    eye = np.eye(dk, dtype=np.float32)
    _, M = _run1(q, k, np.zeros_like(v), g, beta, eye)
    P = np.eye(dk)
    for t in range(7):
        kt = k[t].astype(np.float64)
        P = (np.eye(dk) - float(beta[t]) * np.outer(kt, kt)) @ np.diag(np.exp(g[t].astype(np.float64))) @ P
    assert np.max(np.abs(M - P)) < 1e-12
    q, k, v, g, beta, S0 = _rand_case(40, 8, 8, 32, g_scale=0.5)
    o_full, f_full = _run1(q, k, v, g, beta, S0)
    eye8, zv = np.eye(8, dtype=np.float32), np.zeros_like(v)
    for m in (1, 17, 39):
        _, S_m = _run1(q[:m], k[:m], v[:m], g[:m], beta[:m], S0)
        _, M = _run1(q[m:], k[m:], zv[m:], g[m:], beta[m:], eye8)
        _, S_r = _run1(q[m:], k[m:], v[m:], g[m:], beta[m:], None)
        assert rel_err(M @ S_m + S_r, f_full) < 1e-12
        o_tail, _ = _run1(q[m:], k[m:], v[m:], g[m:], beta[m:], S_m.astype(np.float32))
        assert rel_err(o_tail, o_full[m:]) < 1e-6   # S_m re-enters as fp32
