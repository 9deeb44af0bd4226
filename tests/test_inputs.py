"""The seeded input generator: reproducible draws and the gate recipe."""
import numpy as np

from gated_deltanet_hybrid_gb300.inputs import WORKLOADS, WorkloadStream, gates_from_ab


def test_gate_recipe_against_library():
    a = np.linspace(-40, 40, 161)
    b = np.linspace(-40, 40, 161)
    g, beta = gates_from_ab(a, b)
    assert g.dtype == np.float32 and beta.dtype == np.float32
    assert np.allclose(g, (-0.5 * np.logaddexp(0.0, a)).astype(np.float32), rtol=1e-6, atol=0)
    from scipy.special import expit
    assert np.allclose(beta, expit(b).astype(np.float32), rtol=1e-6, atol=1e-30)
    assert np.all(g <= 0) and np.all((beta >= 0) & (beta <= 1))


def test_streams_are_reproducible():
    s1, s2 = WorkloadStream(WORKLOADS["tiny"]), WorkloadStream(WORKLOADS["tiny"])
    assert np.array_equal(s1.weights[0].w_in, s2.weights[0].w_in)
    for _ in range(3):
        (x1, g1), (x2, g2) = s1.next_step(), s2.next_step()
        assert np.array_equal(x1, x2)
        assert np.array_equal(g1[0][0], g2[0][0]) and np.array_equal(g1[0][1], g2[0][1])


def test_weight_ranges():
    w = WorkloadStream(WORKLOADS["tiny"]).weights[0]
    assert w.w_in.dtype == np.int8 and w.w_in.min() >= -127 and w.w_in.max() <= 127
    assert w.s_in.min() >= 0.001 and w.s_in.max() <= 0.01
    assert w.w_in.shape == (WORKLOADS["tiny"].cfg.in_rows, 256)


def test_decay_band_recipe():
    st = WorkloadStream(WORKLOADS["long_prompt_b8"].__class__(
        "band", WORKLOADS["tiny"].cfg, batch=2, steps=4, seed=4, gate="decay_band"))
    _, gates = st.next_step()
    g, beta = gates[0]
    assert np.all(np.exp(g.astype(np.float64)) >= 0.9 - 1e-7) and np.all(np.exp(g) <= 1.0)
