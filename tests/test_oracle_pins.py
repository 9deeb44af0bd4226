"""Pins for the CPU oracle: each check ties one oracle function to something
other than itself (exact integer arithmetic, a closed form, a hand-worked
case, a brute-force unrolling of the recurrence, or an invariant of the
definition), so that a dropped term, a wrong sign or index or a transposed
operand in the oracle fails here.  CPU only."""
import dataclasses
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle.dn_oracle as dn_oracle
from gated_deltanet_hybrid_gb300.inputs import DNConfig, DNState, DNWeights, make_weights, zero_state
from oracle import (
    OracleLayer,
    gate_transform,
    sigmoid,
    softplus,
    causal_conv_silu_step,
    gated_delta_rule_step,
    gated_rmsnorm,
    int8_rowscaled_gemv,
    l2_normalize,
    rms_prenorm,
    silu,
    stack_step,
)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- int8 GEMV
def test_gemv_exact_integer_case():
    """Integer x in [-3, 3] and power-of-two row scales: every partial sum is
    an exact integer, so the oracle must equal numpy's int64 matmul bitwise."""
    rng = np.random.default_rng(11)
    w = rng.integers(-127, 128, size=(48, 80), dtype=np.int8)          # non-square
    s = (2.0 ** rng.integers(-4, 3, size=48)).astype(np.float32)
    x = rng.integers(-3, 4, size=(5, 80))
    exact = (x.astype(np.int64) @ w.astype(np.int64).T) * s.astype(np.float64)
    got = int8_rowscaled_gemv(w, s, x.astype(np.float32))
    assert got.shape == (5, 48)
    assert np.array_equal(got, exact)


def test_gemv_scale_is_per_output_row():
    w = np.array([[1, 2, 3], [4, 5, 6]], np.int8)
    s = np.array([2.0, 10.0], np.float32)
    got = int8_rowscaled_gemv(w, s, np.array([1.0, 0.0, -1.0], np.float32))
    assert np.array_equal(got, [2.0 * (1 - 3), 10.0 * (4 - 6)])


# ---------------------------------------------------------------- conv + ring
def test_conv_impulse_response_and_ring():
    """A one-hot input at step 0 comes out through tap conv_k-1-t at step t
    (t = 0..conv_k-1) and is gone afterwards; ring_pos counts steps mod
    conv_k-1 and the ring holds the last conv_k-1 inputs."""
    rng = np.random.default_rng(3)
    C, K = 6, 4
    w = rng.uniform(-0.5, 0.5, size=(C, K)).astype(np.float32)
    ring = np.zeros((K - 1, C))
    pos = 0
    inputs = []
    for t in range(9):
        x = np.zeros(C)
        if t == 0:
            x[2] = 1.0
        x_other = rng.standard_normal(C) * (t >= 6)  # later steps: fresh data
        x = x + x_other * (np.arange(C) != 2)
        inputs.append(x.copy())
        u, pos = causal_conv_silu_step(w, ring, pos, x)
        assert pos == (t + 1) % (K - 1)
        if t < K:
            want = float(w[2, K - 1 - t]) * expit(float(w[2, K - 1 - t]))
            assert u[2] == pytest.approx(want, rel=1e-15, abs=1e-300)
        else:
            assert u[2] == 0.0
        # ring: slot (pos + m) mod (K-1), m = 0 oldest .. K-2 newest
        for m in range(K - 1):
            src = t - (K - 2) + m
            want_row = inputs[src] if src >= 0 else np.zeros(C)
            assert np.array_equal(ring[(pos + m) % (K - 1)], want_row)


def test_conv_sums_taps_in_causal_order():
    """Three known past inputs and one current input: the conv output equals
    the hand sum w0*x(t-3) + w1*x(t-2) + w2*x(t-1) + w3*x(t) through SiLU."""
    w = np.array([[1.0, 10.0, 100.0, 1000.0]]) * 1e-3
    ring = np.zeros((3, 1))
    pos = 0
    for val in (1.0, 2.0, 3.0):
        _, pos = causal_conv_silu_step(w, ring, pos, np.array([val]))
    u, pos = causal_conv_silu_step(w, ring, pos, np.array([4.0]))
    pre = 1e-3 * (1 * 1.0 + 10 * 2.0 + 100 * 3.0 + 1000 * 4.0)
    assert u[0] == pytest.approx(pre * expit(pre), rel=1e-14)
    assert pos == 1


def test_silu_against_library_sigmoid():
    x = np.linspace(-30, 30, 121)
    assert np.allclose(silu(x), x * expit(x), rtol=1e-14, atol=0)
    assert silu(np.array([0.0]))[0] == 0.0


# ---------------------------------------------------------------- L2 norm
def test_l2_norm_closed_form():
    eps = 1e-6
    got = l2_normalize(np.array([3.0, 4.0]), eps)
    r = math.sqrt(25.0 + eps)
    assert got[0] == pytest.approx(3.0 / r, rel=1e-15)
    assert got[1] == pytest.approx(4.0 / r, rel=1e-15)
    assert np.allclose(l2_normalize(np.array([3.0, 4.0]), 0.0), [0.6, 0.8], rtol=1e-15)
    assert np.array_equal(l2_normalize(np.zeros(5), eps), np.zeros(5))


# ---------------------------------------------------------------- recurrence
def _golden_2x2():
    vals = {}
    with open(os.path.join(GOLDEN, "handworked_2x2.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *nums = line.split()
            vals[key] = np.array([float(v) for v in nums])
    return vals


def test_handworked_2x2_head():
    gv = _golden_2x2()
    S = np.zeros((2, 2))
    for step in ("step1", "step2"):
        k = l2_normalize(gv[f"{step}.k"], 0.0)
        q = l2_normalize(gv[f"{step}.q"], 0.0)
        g = math.log(gv[f"{step}.decay"][0])
        S, o = gated_delta_rule_step(S, q, k, gv[f"{step}.v"], g, gv[f"{step}.beta"][0])
        assert np.allclose(S.reshape(-1), gv[f"{step}.S"], rtol=0, atol=1e-15)
        assert np.allclose(o, gv[f"{step}.o"], rtol=0, atol=1e-15)


def test_handworked_2x2_head_with_eps():
    gv = _golden_2x2()
    S = np.zeros((2, 2))
    for step in ("step1", "step2"):
        k = l2_normalize(gv[f"{step}.k"], 1e-6)
        q = l2_normalize(gv[f"{step}.q"], 1e-6)
        S, o = gated_delta_rule_step(S, q, k, gv[f"{step}.v"], math.log(gv[f"{step}.decay"][0]),
                                     gv[f"{step}.beta"][0])
        assert np.allclose(S.reshape(-1), gv[f"{step}.S"], atol=3e-6)
        assert np.allclose(o, gv[f"{step}.o"], atol=3e-6)


def test_recurrence_against_unrolled_products():
    """Brute force: with A_t = e^{g_t} (I - beta_t k_t k_t^T),
    S_T = A_T ... A_1 S_0 + sum_s A_T ... A_{s+1} beta_s k_s v_s^T,
    built from explicit dk x dk matrices for 64 steps of a 32x32 head."""
    rng = np.random.default_rng(7)
    dk, dv, T = 32, 24, 64
    S0 = rng.standard_normal((dk, dv)) * 0.1
    ks = [l2_normalize(rng.standard_normal(dk), 1e-6) for _ in range(T)]
    qs = [l2_normalize(rng.standard_normal(dk), 1e-6) for _ in range(T)]
    vs = [rng.standard_normal(dv) for _ in range(T)]
    gs = -0.5 * np.log1p(np.exp(rng.standard_normal(T)))
    bs = expit(rng.standard_normal(T))
    A = [math.exp(gs[t]) * (np.eye(dk) - bs[t] * np.outer(ks[t], ks[t])) for t in range(T)]

    S = S0.copy()
    for t in range(T):
        S, o = gated_delta_rule_step(S, qs[t], ks[t], vs[t], gs[t], bs[t])
        # brute force S_t from scratch
        P = np.eye(dk)
        brute = np.zeros((dk, dv))
        for s in range(t, -1, -1):
            brute = brute + P @ (bs[s] * np.outer(ks[s], vs[s]))
            P = P @ A[s]
        brute = brute + P @ S0
        assert np.allclose(S, brute, rtol=0, atol=1e-12 * max(1.0, np.abs(brute).max()))
        assert np.allclose(o, brute.T @ qs[t], rtol=0, atol=1e-12)


def test_invariant_beta0_decay1_leaves_state():
    rng = np.random.default_rng(1)
    S = rng.standard_normal((16, 8))
    k = l2_normalize(rng.standard_normal(16), 1e-6)
    q = l2_normalize(rng.standard_normal(16), 1e-6)
    S1, o = gated_delta_rule_step(S, q, k, rng.standard_normal(8), 0.0, 0.0)
    assert np.array_equal(S1, S)
    assert np.allclose(o, S.T @ q, rtol=1e-15, atol=1e-15)


def test_invariant_beta0_is_pure_decay():
    rng = np.random.default_rng(2)
    S = rng.standard_normal((16, 8))
    k = l2_normalize(rng.standard_normal(16), 1e-6)
    S1, _ = gated_delta_rule_step(S, k, k, rng.standard_normal(8), -0.3, 0.0)
    assert np.allclose(S1, math.exp(-0.3) * S, rtol=1e-15, atol=0)


def test_invariant_beta1_writes_value_exactly():
    """beta = 1 with a unit key: the updated state maps k to v exactly."""
    rng = np.random.default_rng(4)
    S = rng.standard_normal((16, 8))
    k = rng.standard_normal(16)
    k = k / np.linalg.norm(k)
    v = rng.standard_normal(8)
    S1, _ = gated_delta_rule_step(S, k, k, v, -0.7, 1.0)
    assert np.allclose(S1.T @ k, v, rtol=0, atol=1e-12)


def test_readout_uses_updated_state():
    """q = k, beta = 1, unit k: o = S_new^T k = v, which the pre-update
    state would not give."""
    rng = np.random.default_rng(5)
    S = rng.standard_normal((8, 8))
    k = np.zeros(8)
    k[3] = 1.0
    v = rng.standard_normal(8)
    _, o = gated_delta_rule_step(S, k, k, v, -0.1, 1.0)
    assert np.allclose(o, v, atol=1e-14)


def test_key_gate_handworked_head():
    """Per-key-channel decay scales the rows of S (key index), worked by hand
    in tests/golden/handworked_key_gate.txt."""
    gv = _golden_file("handworked_key_gate.txt")
    S, o = gated_delta_rule_step(gv["S0"].reshape(2, 2), l2_normalize(gv["q"], 0.0),
                                 l2_normalize(gv["k"], 0.0), gv["v"], np.log(gv["decay"]), gv["beta"][0])
    assert np.allclose(S.reshape(-1), gv["S"], rtol=0, atol=1e-15)
    assert np.allclose(o, gv["o"], rtol=0, atol=1e-15)


def test_key_gate_uniform_equals_scalar_gate():
    """A per-key gate with every entry c is the per-head gate c, bitwise."""
    rng = np.random.default_rng(12)
    S = rng.standard_normal((16, 8))
    q = l2_normalize(rng.standard_normal(16), 1e-6)
    k = l2_normalize(rng.standard_normal(16), 1e-6)
    v = rng.standard_normal(8)
    a = gated_delta_rule_step(S, q, k, v, -0.37, 0.6)
    b = gated_delta_rule_step(S, q, k, v, np.full(16, -0.37), 0.6)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_key_gate_recurrence_against_unrolled_products():
    """Brute force with A_t = (I - beta_t k_t k_t^T) diag(exp(g_t)):
    S_T = A_T ... A_1 S_0 + sum_s A_T ... A_{s+1} beta_s k_s v_s^T."""
    rng = np.random.default_rng(13)
    dk, dv, T = 24, 16, 48
    S0 = rng.standard_normal((dk, dv)) * 0.1
    ks = [l2_normalize(rng.standard_normal(dk), 1e-6) for _ in range(T)]
    qs = [l2_normalize(rng.standard_normal(dk), 1e-6) for _ in range(T)]
    vs = [rng.standard_normal(dv) for _ in range(T)]
    gs = -0.5 * np.log1p(np.exp(rng.standard_normal((T, dk))))
    bs = expit(rng.standard_normal(T))
    A = [(np.eye(dk) - bs[t] * np.outer(ks[t], ks[t])) @ np.diag(np.exp(gs[t])) for t in range(T)]
    S = S0.copy()
    for t in range(T):
        S, o = gated_delta_rule_step(S, qs[t], ks[t], vs[t], gs[t], bs[t])
        P = np.eye(dk)
        brute = np.zeros((dk, dv))
        for s in range(t, -1, -1):
            brute = brute + P @ (bs[s] * np.outer(ks[s], vs[s]))
            P = P @ A[s]
        brute = brute + P @ S0
        assert np.allclose(S, brute, rtol=0, atol=1e-12 * max(1.0, np.abs(brute).max()))
        assert np.allclose(o, brute.T @ qs[t], rtol=0, atol=1e-12)


def test_key_gate_layer_uses_each_heads_vector():
    """In a whole layer the per-key gate of (sequence b, head h) reaches that
    head only: zeroing g for one head (decay 1) with beta = 0 leaves exactly
    that head's state unchanged."""
    cfg = DNConfig(hidden=24, n_qk_heads=2, n_v_heads=4, dk=4, dv=4, key_gate=True)
    w = make_weights(cfg, np.random.default_rng(0))
    rng = np.random.default_rng(3)
    st = DNState(S=rng.standard_normal((2, 4, 4, 4)), ring=np.zeros((2, 3, cfg.conv_ch)),
                 ring_pos=np.zeros(2, np.int32))
    layer = OracleLayer(cfg, w, st)
    g = -rng.uniform(0.1, 1.0, (2, 4, 4))
    g[1, 2] = 0.0
    layer.step(rng.standard_normal((2, cfg.hidden)), g, np.zeros((2, 4)))
    for b in range(2):
        for h in range(4):
            want = st.S[b, h] * np.exp(g[b, h])[:, None]
            assert np.allclose(layer.S[b, h], want, rtol=1e-15, atol=0)
    assert np.array_equal(layer.S[1, 2], st.S[1, 2])


# ---------------------------------------------------------------- gated RMSNorm
def test_gated_rmsnorm_invariants():
    rng = np.random.default_rng(6)
    o = rng.standard_normal(128)
    z = rng.standard_normal(128)
    w = rng.uniform(0.5, 1.5, 128)
    a = gated_rmsnorm(o, z, w, 0.0)
    b = gated_rmsnorm(37.5 * o, z, w, 0.0)
    assert np.allclose(a, b, rtol=1e-14, atol=0)
    assert np.array_equal(gated_rmsnorm(o, np.zeros(128), w, 1e-6), np.zeros(128))
    zbig = np.full(128, 60.0)
    want = o / np.sqrt(np.mean(o ** 2)) * 60.0
    assert np.allclose(gated_rmsnorm(o, zbig, np.ones(128), 0.0), want, rtol=1e-14)
    # constant head: every entry normalises to sign(o) (times w * silu(z))
    c = gated_rmsnorm(np.full(4, -2.0), np.full(4, 60.0), np.ones(4), 0.0)
    assert np.allclose(c, -60.0, rtol=1e-14)


def _golden_file(name):
    return _golden(name)


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *nums = line.split()
            vals[key] = np.array([float(v) for v in nums])
    return vals


def _rmsnorm_golden_ok() -> bool:
    """The hand-worked head of tests/golden/handworked_gated_rmsnorm.txt:
    non-uniform weight, z where silu(z) differs from z and from sigmoid(z),
    and an eps whose place (inside or outside the root) changes the result."""
    gv = _golden("handworked_gated_rmsnorm.txt")
    y = dn_oracle.gated_rmsnorm(gv["o"], gv["z"], gv["w"], float(gv["eps"][0]))
    return bool(np.allclose(y, gv["y"], rtol=1e-14, atol=1e-15))


def test_gated_rmsnorm_handworked():
    assert _rmsnorm_golden_ok()


def _hand_layer():
    """The one-head layer of tests/golden/handworked_layer_step.txt, one step."""
    gv = _golden("handworked_layer_step.txt")
    cfg = DNConfig(hidden=8, n_qk_heads=1, n_v_heads=1, dk=2, dv=2, conv_k=2,
                   l2_eps=float(gv["l2_eps"][0]), norm_eps=float(gv["norm_eps"][0]),
                   q_scale=float(gv["q_scale"][0]))
    w_out = np.zeros((8, 2), np.int8)
    w_out[0, 0] = w_out[1, 1] = 1
    w = DNWeights(w_in=np.eye(8, dtype=np.int8), s_in=np.ones(8, np.float32),
                  w_conv=np.tile(np.array([0.0, 1.0], np.float32), (cfg.conv_ch, 1)),
                  w_norm=gv["w_norm"].astype(np.float32), w_out=w_out, s_out=np.ones(8, np.float32))
    st = DNState(S=gv["S0"].reshape(1, 1, 2, 2), ring=np.zeros((1, 1, cfg.conv_ch)),
                 ring_pos=np.zeros(1, np.int32))
    layer = OracleLayer(cfg, w, st)
    tr = {}
    out = layer.step(gv["x"].reshape(1, 8), np.array([[math.log(gv["decay"][0])]]),
                     np.array([[gv["beta"][0]]]), trace=tr)
    return out, layer, tr, gv


def _layer_golden_ok() -> bool:
    out, layer, tr, gv = _hand_layer()
    return bool(np.allclose(layer.S[0, 0].reshape(-1), gv["S"], rtol=0, atol=1e-14)
                and np.allclose(tr["o"][0, 0], gv["o"], rtol=0, atol=1e-14)
                and np.allclose(out[0], gv["out"], rtol=0, atol=1e-14))


def test_layer_step_handworked():
    """A whole step of a one-head layer worked by hand: the readout uses
    q_scale times the normalised q, the gated RMSNorm (norm_eps = 1, large
    enough that the scale of o shows) and the out_proj."""
    assert _layer_golden_ok()
    _, layer, _, gv = _hand_layer()
    assert layer.ring_pos[0] == 0  # one slot: the position stays 0
    assert np.array_equal(layer.ring[0, 0], gv["x"][:6])


# Planted mistakes: each is a plausible error in the oracle; the pins above
# must catch every one of them (the mutation is undone after each case).
def _silu(z):
    return z / (1.0 + np.exp(-z))


RMSNORM_MUTANTS = {
    "weight dropped": lambda o, z, w, eps: o / np.sqrt(np.mean(o * o) + eps) * _silu(z),
    "gated by z": lambda o, z, w, eps: o / np.sqrt(np.mean(o * o) + eps) * w * z,
    "gated by sigmoid(z)": lambda o, z, w, eps: o / np.sqrt(np.mean(o * o) + eps) * w / (1 + np.exp(-z)),
    "eps outside the root": lambda o, z, w, eps: o / (np.sqrt(np.mean(o * o)) + eps) * w * _silu(z),
    "sum for mean": lambda o, z, w, eps: o / np.sqrt(np.sum(o * o) + eps) * w * _silu(z),
}


@pytest.mark.parametrize("name", sorted(RMSNORM_MUTANTS))
def test_pins_catch_rmsnorm_mutant(name, monkeypatch):
    monkeypatch.setattr(dn_oracle, "gated_rmsnorm",
                        lambda o, z, w, eps: RMSNORM_MUTANTS[name](np.asarray(o, np.float64),
                                                                   np.asarray(z, np.float64),
                                                                   np.asarray(w, np.float64), eps))
    assert not (_rmsnorm_golden_ok() and _layer_golden_ok())


QSCALE_MUTANTS = {
    "q_scale on k": lambda q, k, e, s: (dn_oracle.l2_normalize(q, e), dn_oracle.l2_normalize(k, e) * s),
    "q_scale before the norm": lambda q, k, e, s: (dn_oracle.l2_normalize(q * s, e), dn_oracle.l2_normalize(k, e)),
    "q_scale dropped": lambda q, k, e, s: (dn_oracle.l2_normalize(q, e), dn_oracle.l2_normalize(k, e)),
    "q and k swapped": lambda q, k, e, s: (dn_oracle.l2_normalize(k, e) * s, dn_oracle.l2_normalize(q, e)),
}


@pytest.mark.parametrize("name", sorted(QSCALE_MUTANTS))
def test_pins_catch_qscale_mutant(name, monkeypatch):
    monkeypatch.setattr(dn_oracle, "normalize_qk", QSCALE_MUTANTS[name])
    assert not _layer_golden_ok()


# ---------------------------------------------------------------- gate transform
def test_softplus_closed_forms_and_library():
    assert softplus(np.array(0.0)) == pytest.approx(math.log(2.0), rel=1e-16)
    x = np.linspace(-30, 30, 241)
    assert np.allclose(softplus(x) - softplus(-x), x, rtol=0, atol=1e-13)   # softplus(x) - softplus(-x) = x
    assert np.allclose(softplus(x), np.logaddexp(0.0, x), rtol=1e-14, atol=0)
    assert softplus(np.array(40.0)) == pytest.approx(40.0, rel=1e-16)
    assert softplus(np.array(-40.0)) == pytest.approx(math.exp(-40.0), rel=1e-12)
    assert softplus(np.array(-800.0)) == 0.0 and softplus(np.array(800.0)) == 800.0


def test_sigmoid_closed_forms_and_library():
    assert sigmoid(np.array(0.0)) == 0.5
    assert sigmoid(np.array(math.log(3.0))) == pytest.approx(0.75, rel=1e-15)
    x = np.linspace(-40, 40, 161)
    assert np.allclose(sigmoid(x) + sigmoid(-x), 1.0, rtol=0, atol=1e-15)
    assert np.allclose(sigmoid(x), expit(x), rtol=1e-14, atol=0)


def test_gate_transform_handworked():
    """a = (0, ln(e - 1)) -> softplus = (ln 2, 1); A = (0.5, 2) ->
    g = (-0.5 ln 2, -2); b = (0, ln 3) -> beta = (0.5, 0.75).  With a per-key
    gate each head's coefficient multiplies all of its dk values."""
    a = np.array([[0.0, math.log(math.e - 1.0)]])
    b = np.array([[0.0, math.log(3.0)]])
    g, beta = gate_transform(a, b, np.array([0.5, 2.0]))
    assert np.allclose(g, [[-0.5 * math.log(2.0), -2.0]], rtol=1e-15, atol=0)
    assert np.allclose(beta, [[0.5, 0.75]], rtol=1e-15, atol=0)
    ak = np.stack([np.zeros(3), np.full(3, math.log(math.e - 1.0))])[None]  # [1][2 heads][dk 3]
    gk, _ = gate_transform(ak, b, np.array([0.5, 2.0]))
    assert np.allclose(gk[0, 0], -0.5 * math.log(2.0), rtol=1e-15) and np.allclose(gk[0, 1], -2.0, rtol=1e-15)


@pytest.mark.parametrize("key_gate", [False, True])
def test_device_gates_are_the_a_b_rows_of_the_layer(key_gate):
    """A layer with device gates steps exactly like the same layer given
    host gates computed from its a rows (n_v * gate_width, first) and b rows
    (n_v, after them) by an exact integer product and the pinned transform."""
    cfg = DNConfig(hidden=24, n_qk_heads=2, n_v_heads=4, dk=4, dv=4, key_gate=key_gate, device_gates=True)
    w = make_weights(cfg, np.random.default_rng(4))
    rng = np.random.default_rng(5)
    dev = OracleLayer(cfg, w, zero_state(cfg, 2))
    host = OracleLayer(dataclasses.replace(cfg, device_gates=False), w, zero_state(cfg, 2))
    for _ in range(3):
        x = rng.integers(-3, 4, size=(2, cfg.hidden)).astype(np.float64)
        ab = (x.astype(np.int64) @ w.w_ab.astype(np.int64).T) * w.s_ab.astype(np.float64)
        na = cfg.n_v_heads * cfg.gate_width
        a = ab[:, :na].reshape((2, 4, 4) if key_gate else (2, 4))
        g, beta = gate_transform(a, ab[:, na:], w.gate_A)
        out_d = dev.step(x)
        out_h = host.step(x, g, beta)
        assert np.allclose(out_d, out_h, rtol=1e-13, atol=1e-13)
    assert np.allclose(dev.S, host.S, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- whole step
TINY2 = DNConfig(hidden=24, n_qk_heads=2, n_v_heads=4, dk=4, dv=4)


def _tiny_layer(cfg=TINY2, seed=0):
    w = make_weights(cfg, np.random.default_rng(seed))
    return w, OracleLayer(cfg, w, zero_state(cfg, 1))


def test_step_channel_layout_v_block():
    """Zeroing the in_proj rows of v head 1 keeps that head's state at zero
    (v = silu(conv(0)) = 0, so delta = 0) while every other head fills."""
    cfg = TINY2
    w = make_weights(cfg, np.random.default_rng(0))
    v0 = 2 * cfg.qk_dim
    w.w_in[v0 + 1 * cfg.dv: v0 + 2 * cfg.dv] = 0
    layer = OracleLayer(cfg, w, zero_state(cfg, 1))
    rng = np.random.default_rng(1)
    for _ in range(3):
        layer.step(rng.standard_normal((1, cfg.hidden)), np.full((1, 4), -0.2), np.full((1, 4), 0.7))
    norms = [np.abs(layer.S[0, h]).max() for h in range(4)]
    assert norms[1] == 0.0 and min(norms[0], norms[2], norms[3]) > 0.0


def test_step_channel_layout_k_block_and_head_sharing():
    """Zeroing the k rows of q/k head 0 leaves value heads 0 and 1 (which
    share it) with zero state; heads 2 and 3 read q/k head 1 and fill."""
    cfg = TINY2
    w = make_weights(cfg, np.random.default_rng(0))
    w.w_in[cfg.qk_dim: cfg.qk_dim + cfg.dk] = 0
    layer = OracleLayer(cfg, w, zero_state(cfg, 1))
    rng = np.random.default_rng(2)
    for _ in range(3):
        layer.step(rng.standard_normal((1, cfg.hidden)), np.full((1, 4), -0.2), np.full((1, 4), 0.7))
    norms = [np.abs(layer.S[0, h]).max() for h in range(4)]
    assert norms[0] == 0.0 and norms[1] == 0.0
    assert norms[2] > 0.0 and norms[3] > 0.0


def test_step_channel_layout_q_and_z_blocks():
    """Zero q rows of q/k head 1 -> readout of value heads 2, 3 is zero;
    zero z rows of value head 0 -> its normed output is zero (silu(0) = 0)."""
    cfg = TINY2
    w = make_weights(cfg, np.random.default_rng(0))
    w.w_in[1 * cfg.dk: 2 * cfg.dk] = 0
    z0 = cfg.conv_ch
    w.w_in[z0: z0 + cfg.dv] = 0
    layer = OracleLayer(cfg, w, zero_state(cfg, 1))
    rng = np.random.default_rng(3)
    tr = {}
    for _ in range(3):
        layer.step(rng.standard_normal((1, cfg.hidden)), np.full((1, 4), -0.2), np.full((1, 4), 0.7), trace=tr)
    o = tr["o"][0]
    assert np.all(o[2] == 0.0) and np.all(o[3] == 0.0)
    assert np.abs(o[0]).max() > 0 and np.abs(o[1]).max() > 0
    n = tr["normed"][0]
    assert np.all(n[0:cfg.dv] == 0.0) and np.abs(n[cfg.dv:]).max() > 0


def test_step_conv_impulse_through_in_proj():
    """A hand-set in_proj routes x[5] alone to conv channel c with weight 1
    (scale 1); a one-hot x then shows silu(w_conv[c][K-1-t]) at channel c
    of the conv output for t = 0..K-1 and nothing after."""
    cfg = TINY2
    w = make_weights(cfg, np.random.default_rng(0))
    c = 2 * cfg.qk_dim + 3  # a v channel
    w.w_in[:] = 0
    w.w_in[c, 5] = 1
    w.s_in[:] = 1.0
    layer = OracleLayer(cfg, w, zero_state(cfg, 1))
    for t in range(cfg.conv_k + 2):
        x = np.zeros((1, cfg.hidden))
        if t == 0:
            x[0, 5] = 1.0
        tr = {}
        layer.step(x, np.zeros((1, 4)), np.zeros((1, 4)), trace=tr)
        u = tr["u"][0]
        if t < cfg.conv_k:
            wt = float(w.w_conv[c, cfg.conv_k - 1 - t])
            assert u[c] == pytest.approx(wt * expit(wt), rel=1e-14)
        else:
            assert u[c] == 0.0
        assert np.count_nonzero(u) <= 1
        assert layer.ring_pos[0] == (t + 1) % (cfg.conv_k - 1)


def test_step_batch_rows_are_independent():
    """Sequences share weights only: stepping a batch of three equals
    stepping each sequence alone."""
    cfg = TINY2
    w = make_weights(cfg, np.random.default_rng(9))
    rng = np.random.default_rng(10)
    st = DNState(S=(rng.standard_normal((3, 4, 4, 4)) * 0.1).astype(np.float32),
                 ring=(rng.standard_normal((3, 3, cfg.conv_ch)) * 0.1).astype(np.float32),
                 ring_pos=np.array([0, 1, 2], np.int32))
    batch = OracleLayer(cfg, w, st)
    singles = [OracleLayer(cfg, w, DNState(st.S[b:b + 1], st.ring[b:b + 1], st.ring_pos[b:b + 1]))
               for b in range(3)]
    for _ in range(4):
        x = rng.standard_normal((3, cfg.hidden))
        g = -rng.uniform(0, 1, (3, 4))
        be = rng.uniform(0, 1, (3, 4))
        out = batch.step(x, g, be)
        for b in range(3):
            ob = singles[b].step(x[b:b + 1], g[b:b + 1], be[b:b + 1])
            # a batched matmul may round differently from a single row
            assert np.allclose(out[b], ob[0], rtol=1e-12, atol=1e-12)
    for b in range(3):
        assert np.allclose(batch.S[b], singles[b].S[0], rtol=1e-12, atol=1e-12)
        assert np.allclose(batch.ring[b], singles[b].ring[0], rtol=1e-12, atol=1e-12)
        assert batch.ring_pos[b] == singles[b].ring_pos[0]


# ---------------------------------------------------------------- stack
def test_rms_prenorm_closed_form():
    x = np.array([[3.0, -3.0, 3.0, -3.0], [1.0, 2.0, 2.0, 4.0]])
    got = rms_prenorm(x, 0.0)
    assert np.allclose(got[0], [1, -1, 1, -1], rtol=1e-15)
    assert np.allclose(got[1], np.array([1, 2, 2, 4]) / math.sqrt(25 / 4), rtol=1e-15)


def test_stack_is_residual():
    """A layer whose out_proj is zero passes x through unchanged."""
    cfg = TINY2
    w = make_weights(cfg, np.random.default_rng(0))
    w.w_out[:] = 0
    layers = [OracleLayer(cfg, w, zero_state(cfg, 2)) for _ in range(3)]
    x = np.random.default_rng(1).standard_normal((2, cfg.hidden))
    gates = [(np.full((2, 4), -0.1), np.full((2, 4), 0.5))] * 3
    assert np.array_equal(stack_step(layers, x, gates), x)
