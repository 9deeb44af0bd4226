"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs.  Bar: max|gpu - ref| / max|ref| <= 2e-3 for the
outputs at every step and for the state S and the conv ring at every
checkpoint; the ring positions equal exactly."""
import numpy as np
import pytest

from gated_deltanet_hybrid_gb300.inputs import (SHAPE_35B, TINY, WORKLOADS, DNConfig,
                                                custom_workload)

from harness import REL_TOL, run_parity

pytestmark = pytest.mark.gpu


def _assert_ok(w):
    assert w["out"] <= REL_TOL, w
    assert w["S"] <= REL_TOL, w
    assert w["ring"] <= REL_TOL, w
    assert w["ring_pos_equal"], w


def test_tiny_64_steps():
    _assert_ok(run_parity(WORKLOADS["tiny"]))


def test_35b_batch1_256_steps():
    _assert_ok(run_parity(WORKLOADS["35b_b1"]))


def test_35b_batch64_256_steps_sampled():
    """All 64 sequences run on the GPU; 8 of them (spread over the batch,
    including the last) are recomputed by the oracle."""
    sample = np.array([0, 9, 18, 27, 36, 45, 54, 63])
    _assert_ok(run_parity(WORKLOADS["35b_b64"], sample=sample))


def test_long_prompt_2048_steps_sampled():
    """Batch 8, 2048 tokens with exp(g) in [0.9, 1]: drift against the
    oracle checked at steps 512, 1024 and 2048 on sequences 0 and 7."""
    _assert_ok(run_parity(WORKLOADS["long_prompt_b8"], sample=np.array([0, 7])))


@pytest.mark.parametrize("batch", [2, 3, 5, 16])
def test_35b_small_batches(batch):
    """Batches that take the split-column path (2..4 slices per head, one
    cluster per head) and the NB-chunked GEMV with a ragged last chunk."""
    wl = custom_workload(f"35b_b{batch}", SHAPE_35B, batch=batch, steps=12, seed=20 + batch,
                         init_std=0.02)
    _assert_ok(run_parity(wl, sample=np.array(sorted({0, batch - 1}))))


@pytest.mark.parametrize("dims", [
    dict(hidden=64, n_qk_heads=1, n_v_heads=1, dk=32, dv=32, conv_k=2),
    dict(hidden=128, n_qk_heads=2, n_v_heads=8, dk=64, dv=32, conv_k=5),
    dict(hidden=96, n_qk_heads=3, n_v_heads=3, dk=32, dv=128, conv_k=4),
    dict(hidden=512, n_qk_heads=2, n_v_heads=4, dk=128, dv=64, conv_k=3),
    dict(hidden=256, n_qk_heads=1, n_v_heads=4, dk=64, dv=128, conv_k=4, q_scale=1.0),
])
def test_other_dimensions(dims):
    cfg = DNConfig(**dims)
    wl = custom_workload("dims", cfg, batch=3, steps=20, seed=5, init_std=0.05)
    _assert_ok(run_parity(wl))


def test_tiny_ragged_batch_in_larger_layer():
    """A layer sized for 7 sequences stepping 5 of them: the parity of the
    5, and the untouched 2 keep their state (checked in the layer tests)."""
    wl = custom_workload("tiny_b5", TINY, batch=5, steps=30, seed=8, init_std=0.1)
    _assert_ok(run_parity(wl, max_batch=7))


@pytest.mark.parametrize("batch", [1, 3, 8, 20])
def test_35b_small_batch_in_a_layer_sized_for_64(batch):
    """A layer sized for 64 sequences stepping fewer: the projections'
    schedules (and so their segment counts) depend on the batch, and the
    layer's scratch must hold the largest of them (batch 1 runs the most
    segments per tile)."""
    wl = custom_workload("b%d_in_64" % batch, SHAPE_35B, batch=batch, steps=6, seed=31 + batch,
                         init_std=0.02)
    _assert_ok(run_parity(wl, sample=np.array(sorted({0, batch - 1})), max_batch=64))


@pytest.mark.parametrize("batch", [2, 3, 8, 9, 40, 64, 65, 130])
def test_tiny_tensor_core_batches(batch):
    """Batches from 2 take the tensor-core projections: padded batch columns
    (2, 3 -> 8; 9 -> 16), several 64-sequence chunks (65, 130) and split-K
    tiles."""
    wl = custom_workload(f"tiny_b{batch}", TINY, batch=batch, steps=10, seed=30 + batch, init_std=0.05)
    sample = np.array(sorted({0, batch // 2, batch - 1}))
    _assert_ok(run_parity(wl, sample=sample))


def test_35b_largest_accepted_batch():
    """max_batch = 1024, the largest a layer accepts: 16 batch chunks in the
    tensor-core projections, 216 items per CTA in the state kernel; three
    sequences (first, middle, last) recomputed by the oracle."""
    wl = custom_workload("35b_b1024", SHAPE_35B, batch=1024, steps=3, seed=1024, init_std=0.0)
    _assert_ok(run_parity(wl, sample=np.array([0, 517, 1023])))


def test_tiny_largest_accepted_batch():
    wl = custom_workload("tiny_b1024", TINY, batch=1024, steps=6, seed=77, init_std=0.1)
    _assert_ok(run_parity(wl, sample=np.array([0, 1, 500, 1022, 1023])))


def test_35b_batch65_two_chunks():
    wl = custom_workload("35b_b65", SHAPE_35B, batch=65, steps=6, seed=65, init_std=0.02)
    _assert_ok(run_parity(wl, sample=np.array([0, 63, 64])))


@pytest.mark.parametrize("batch", [1, 3, 8, 37, 64])
def test_in_proj_exact_integer_case(batch):
    """Integer x in [-3, 3] and power-of-two row scales make every partial
    sum of the in_proj an exact integer below 2^24, on the CUDA cores and on
    the tensor cores alike.  After one step the ring holds the in_proj's q|k|v
    rows, which must then equal numpy's int64 matmul bitwise."""
    import torch
    from gated_deltanet_hybrid_gb300 import abi
    from gated_deltanet_hybrid_gb300.inputs import make_weights
    from harness import GpuLayer

    cfg = SHAPE_35B
    rng = np.random.default_rng(100 + batch)
    w = make_weights(cfg, rng)
    w.s_in[:] = (2.0 ** rng.integers(-3, 2, size=cfg.in_rows)).astype(np.float32)
    x = rng.integers(-3, 4, size=(batch, cfg.hidden)).astype(np.float32)
    exact = (x.astype(np.int64) @ w.w_in.astype(np.int64).T) * w.s_in.astype(np.float64)
    layer = GpuLayer.create(cfg, w, batch)
    try:
        out = torch.empty((batch, cfg.hidden), device="cuda")
        g = torch.zeros((batch, cfg.n_v_heads), device="cuda")
        abi.dn_step(layer.handle, batch, torch.from_numpy(x).cuda(), g, g.clone(), out)
        st = layer.get_state()
        # ring_pos 0 -> 1 after one step: the newest input sits in slot 0
        newest = st.ring[:, 0, :]
        assert np.array_equal(newest.astype(np.float64), exact[:, :cfg.conv_ch])
        assert np.all(st.ring_pos == 1)
    finally:
        layer.destroy()


# ---- other dimensions and gates of the same step (48 value heads, head sizes
#      up to 256, the per-key-channel gate of the page's KDA engines) --------
SHAPE_48V = DNConfig(hidden=2048, n_qk_heads=16, n_v_heads=48, dk=128, dv=128)


@pytest.mark.parametrize("batch", [1, 8, 64])
def test_48_value_heads(batch):
    """Three value heads per q/k head (16 q/k heads, 48 value heads of 128):
    the CUDA-core and the tensor-core projections (in_proj 2048 -> 16384,
    out_proj 6144 -> 2048) and the streaming state kernel."""
    wl = custom_workload(f"v48_b{batch}", SHAPE_48V, batch=batch, steps=16, seed=480 + batch, init_std=0.02)
    _assert_ok(run_parity(wl, sample=np.array(sorted({0, batch // 2, batch - 1}))))


@pytest.mark.parametrize("dims", [
    dict(hidden=512, n_qk_heads=2, n_v_heads=4, dk=256, dv=256),
    dict(hidden=256, n_qk_heads=1, n_v_heads=2, dk=256, dv=128, conv_k=3),
    dict(hidden=256, n_qk_heads=2, n_v_heads=2, dk=128, dv=256, conv_k=2),
    dict(hidden=128, n_qk_heads=1, n_v_heads=3, dk=32, dv=256),
    dict(hidden=256, n_qk_heads=2, n_v_heads=4, dk=256, dv=32),
])
@pytest.mark.parametrize("batch", [1, 3, 16])
def test_head_sizes_up_to_256(dims, batch):
    cfg = DNConfig(**dims)
    wl = custom_workload("d256", cfg, batch=batch, steps=16, seed=256 + batch, init_std=0.05)
    _assert_ok(run_parity(wl, sample=np.array(sorted({0, batch - 1}))))


@pytest.mark.parametrize("dims,batch", [
    (dict(hidden=256, n_qk_heads=2, n_v_heads=4, dk=32, dv=32), 3),
    (dict(hidden=512, n_qk_heads=2, n_v_heads=4, dk=256, dv=128), 9),
    (dict(hidden=2048, n_qk_heads=16, n_v_heads=32, dk=128, dv=128), 1),
    (dict(hidden=2048, n_qk_heads=16, n_v_heads=32, dk=128, dv=128), 64),
])
def test_key_gate(dims, batch):
    """The per-key-channel gate on the generic state kernel (32 and 256-wide
    keys) and on the streaming one (128 x 128 heads, batch 1 and 64)."""
    cfg = DNConfig(key_gate=True, **dims)
    wl = custom_workload("kgate", cfg, batch=batch, steps=24, seed=700 + batch, init_std=0.02)
    _assert_ok(run_parity(wl, sample=np.array(sorted({0, batch - 1}))))


def test_key_gate_35b_batch16_256_steps():
    """A per-key-gate workload of the 35B-shape layer at batch 16 over 256
    steps (exp(g) per key row in [0.9, 1], so the state keeps a long memory),
    with the state and ring compared at steps 64 and 256."""
    cfg = DNConfig(hidden=2048, n_qk_heads=16, n_v_heads=32, dk=128, dv=128, key_gate=True)
    wl = custom_workload("kgate_35b_b16", cfg, batch=16, steps=256, seed=716, init_std=0.02, gate="decay_band")
    _assert_ok(run_parity(wl, sample=np.array([0, 15]), checkpoints=(64, 256)))


# ---- device-side gates: the a/b gate projections as int8 rows of the layer --
@pytest.mark.parametrize("batch", [1, 8, 64])
def test_device_gates_35b(batch):
    """The a/b gate rows ride in the in_proj (CUDA-core and tensor-core
    projections, 12288 + 64 rows) and the streaming state kernel turns them
    into the decay and the write strength."""
    cfg = DNConfig(hidden=2048, n_qk_heads=16, n_v_heads=32, dk=128, dv=128, device_gates=True)
    wl = custom_workload(f"devg_b{batch}", cfg, batch=batch, steps=32, seed=900 + batch, init_std=0.02)
    _assert_ok(run_parity(wl, sample=np.array(sorted({0, batch - 1}))))


@pytest.mark.parametrize("dims,batch", [
    (dict(hidden=256, n_qk_heads=2, n_v_heads=4, dk=32, dv=32), 3),
    (dict(hidden=256, n_qk_heads=2, n_v_heads=4, dk=32, dv=32, key_gate=True), 9),
    (dict(hidden=512, n_qk_heads=2, n_v_heads=4, dk=256, dv=128, key_gate=True), 2),
    (dict(hidden=2048, n_qk_heads=16, n_v_heads=32, dk=128, dv=128, key_gate=True), 16),
])
def test_device_gates_other_shapes(dims, batch):
    """Device gates on the generic state kernel (32- and 256-wide keys), with
    one gate per head and with the per-key gate (a rows per key channel), and
    on the streaming kernel with the per-key gate."""
    cfg = DNConfig(device_gates=True, **dims)
    wl = custom_workload("devg", cfg, batch=batch, steps=24, seed=950 + batch, init_std=0.02)
    _assert_ok(run_parity(wl, sample=np.array(sorted({0, batch - 1}))))


def test_device_gates_reject_host_gates():
    """A layer with device gates refuses g / beta, and a layer without them
    refuses NULL gates, before any device work."""
    import torch
    from gated_deltanet_hybrid_gb300 import abi
    from gated_deltanet_hybrid_gb300.inputs import make_weights
    from harness import GpuLayer

    for dev in (True, False):
        cfg = DNConfig(hidden=256, n_qk_heads=2, n_v_heads=4, dk=32, dv=32, device_gates=dev)
        layer = GpuLayer.create(cfg, make_weights(cfg, np.random.default_rng(1)), 2)
        try:
            x = torch.zeros((2, 256), device="cuda")
            out = torch.empty_like(x)
            g = torch.zeros((2, 4), device="cuda")
            if dev:
                assert abi.dn_step(layer.handle, 2, x, g, g, out, check=False) == abi.DN_EINVAL
            else:
                assert abi.dn_step(layer.handle, 2, x, None, None, out, check=False) == abi.DN_EINVAL
        finally:
            layer.destroy()


# ---- per-row int4 weights (the page's model container) -----------------------
SHAPE_35B_I4 = DNConfig(hidden=2048, n_qk_heads=16, n_v_heads=32, dk=128, dv=128, int4=True)


@pytest.mark.parametrize("batch", [1, 3, 8, 64])
def test_int4_weights_35b(batch):
    """int4 weights: the CUDA-core GEMV streams the packed int4 tiles (batch
    1), the tensor-core projections their exact int8 expansion (3, 8, 64)."""
    wl = custom_workload(f"i4_b{batch}", SHAPE_35B_I4, batch=batch, steps=24, seed=440 + batch, init_std=0.02)
    _assert_ok(run_parity(wl, sample=np.array(sorted({0, batch - 1}))))


@pytest.mark.parametrize("batch", [1, 2])
def test_int4_with_device_gates_and_odd_sizes(batch):
    """int4 in_proj with the a/b gate rows appended (16 + 64 rows past the
    q|k|v|z rows), a hidden size that is not a multiple of 128, batch 1
    (the int4 GEMV) and 2 (the tensor cores on the int8 expansion)."""
    cfg = DNConfig(hidden=208, n_qk_heads=2, n_v_heads=4, dk=64, dv=64, int4=True, device_gates=True)
    wl = custom_workload("i4_odd", cfg, batch=batch, steps=20, seed=443 + batch, init_std=0.05)
    _assert_ok(run_parity(wl))


@pytest.mark.parametrize("batch", [1, 5])
def test_int4_in_proj_exact_integer_case(batch):
    """Integer x in [-3, 3], int4 weights and power-of-two row scales: every
    partial sum is an exact integer, so the ring's newest slot (the in_proj's
    q|k|v rows) equals numpy's int64 matmul bitwise."""
    import torch
    from gated_deltanet_hybrid_gb300 import abi
    from gated_deltanet_hybrid_gb300.inputs import make_weights
    from harness import GpuLayer

    cfg = SHAPE_35B_I4
    rng = np.random.default_rng(200 + batch)
    w = make_weights(cfg, rng)
    w.s_in[:] = (2.0 ** rng.integers(-3, 2, size=cfg.in_rows)).astype(np.float32)
    x = rng.integers(-3, 4, size=(batch, cfg.hidden)).astype(np.float32)
    exact = (x.astype(np.int64) @ w.w_in.astype(np.int64).T) * w.s_in.astype(np.float64)
    layer = GpuLayer.create(cfg, w, batch)
    try:
        out = torch.empty((batch, cfg.hidden), device="cuda")
        g = torch.zeros((batch, cfg.n_v_heads), device="cuda")
        abi.dn_step(layer.handle, batch, torch.from_numpy(x).cuda(), g, g.clone(), out)
        newest = layer.get_state().ring[:, 0, :]
        assert np.array_equal(newest.astype(np.float64), exact[:, :cfg.conv_ch])
    finally:
        layer.destroy()
