"""The layer object's contract on the GPU: state ownership (set/get round
trip, slices, ring-position convention), failure handling (as with the page's fake
backend: a step can be made to fail, the failure switches the layer off and
the host carries on from the state read back from the card), device-memory accounting, bitwise
reproducibility and checkpoint/resume."""
import numpy as np
import pytest

from gated_deltanet_hybrid_gb300 import abi
from gated_deltanet_hybrid_gb300.inputs import (SHAPE_35B, TINY, DNState, WorkloadStream,
                                                custom_workload, make_weights, random_state)

from harness import GpuLayer

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


def _dev_inputs(x, g, b):
    torch = _torch()
    return (torch.from_numpy(x).cuda(), torch.from_numpy(g).cuda(), torch.from_numpy(b).cuda(),
            torch.empty(x.shape, dtype=torch.float32, device="cuda"))


def _run(layer, stream, steps, batch):
    outs = []
    for _ in range(steps):
        x, gates = stream.next_step()
        xd, gd, bd, od = _dev_inputs(x[:batch], gates[0][0][:batch], gates[0][1][:batch])
        abi.dn_step(layer.handle, batch, xd, gd, bd, od)
        outs.append(od.cpu().numpy())
    return outs


def test_state_round_trip_is_exact_host_and_device():
    torch = _torch()
    rng = np.random.default_rng(0)
    w = make_weights(TINY, rng)
    st = random_state(TINY, 6, rng, 0.5)
    st.ring_pos[:] = [0, 1, 2, 2, 1, 0]
    layer = GpuLayer.create(TINY, w, 6, st)
    try:
        back = layer.get_state()
        assert np.array_equal(back.S, st.S)
        assert np.array_equal(back.ring, st.ring)
        assert np.array_equal(back.ring_pos, st.ring_pos)
        # slice [2, 5) through device pointers
        S_d = torch.empty((3, 4, 32, 32), dtype=torch.float32, device="cuda")
        r_d = torch.empty((3, 3, TINY.conv_ch), dtype=torch.float32, device="cuda")
        p_d = torch.empty(3, dtype=torch.int32, device="cuda")
        abi.dn_get_state(layer.handle, 2, 3, S_d, r_d, p_d)
        assert np.array_equal(S_d.cpu().numpy(), st.S[2:5])
        assert np.array_equal(r_d.cpu().numpy(), st.ring[2:5])
        assert np.array_equal(p_d.cpu().numpy(), st.ring_pos[2:5])
        # push a modified slice back through device pointers
        abi.dn_set_state(layer.handle, 0, S_d * 2, r_d + 1, torch.tensor([1, 1, 1], dtype=torch.int32,
                                                                          device="cuda"))
        back2 = layer.get_state()
        assert np.array_equal(back2.S[:3], st.S[2:5] * 2)
        assert np.array_equal(back2.ring[:3], st.ring[2:5] + 1)
        assert list(back2.ring_pos[:3]) == [1, 1, 1]
        assert np.array_equal(back2.S[3:], st.S[3:])
    finally:
        layer.destroy()


def test_ring_positions_advance_after_set_state():
    """ring_pos set to p advances to (p + t) mod (conv_k-1) after t steps, and
    the ring then holds exactly the last conv_k-1 in_proj outputs."""
    rng = np.random.default_rng(1)
    w = make_weights(TINY, rng)
    st = random_state(TINY, 3, rng, 0.1)
    st.ring_pos[:] = [2, 0, 1]
    layer = GpuLayer.create(TINY, w, 3, st)
    try:
        stream = WorkloadStream(custom_workload("t", TINY, 3, 5, seed=3))
        _run(layer, stream, 5, 3)
        assert list(layer.get_state().ring_pos) == [(2 + 5) % 3, (0 + 5) % 3, (1 + 5) % 3]
    finally:
        layer.destroy()


def test_invalid_arguments_leave_state_untouched():
    torch = _torch()
    rng = np.random.default_rng(2)
    w = make_weights(TINY, rng)
    st = random_state(TINY, 2, rng, 0.3)
    layer = GpuLayer.create(TINY, w, 2, st)
    try:
        bad = st.ring_pos.copy()
        bad[1] = 3  # conv_k - 1 slots: valid values 0..2
        rc = abi.dn_set_state(layer.handle, 0, st.S * 0, st.ring * 0, bad, check=False)
        assert rc == abi.DN_EINVAL
        x = torch.zeros((3, 256), device="cuda")
        g = torch.zeros((3, 4), device="cuda")
        rc = abi.dn_step(layer.handle, 3, x, g, g, x.clone(), check=False)  # batch > max_batch
        assert rc == abi.DN_EINVAL
        rc = abi.dn_step(layer.handle, 0, x, g, g, x.clone(), check=False)  # empty batch
        assert rc == abi.DN_EINVAL
        assert abi.dn_get_state(layer.handle, 1, 2, np.empty((2, 4, 32, 32), np.float32),
                                check=False) == abi.DN_EINVAL
        back = layer.get_state()
        assert np.array_equal(back.S, st.S) and np.array_equal(back.ring, st.ring)
        assert np.array_equal(back.ring_pos, st.ring_pos)
    finally:
        layer.destroy()


def test_injected_failure_turns_layer_off_and_state_stays_readable():
    rng = np.random.default_rng(3)
    w = make_weights(TINY, rng)
    layer = GpuLayer.create(TINY, w, 2)
    try:
        stream = WorkloadStream(custom_workload("t", TINY, 2, 8, seed=4))
        _run(layer, stream, 4, 2)
        good = layer.get_state()
        abi.dn_debug_fail_next(layer.handle, abi.DN_EINJECTED)
        x, gates = stream.next_step()
        xd, gd, bd, od = _dev_inputs(x, *gates[0])
        assert abi.dn_step(layer.handle, 2, xd, gd, bd, od, check=False) == abi.DN_EINJECTED
        assert abi.dn_step(layer.handle, 2, xd, gd, bd, od, check=False) == abi.DN_EFAILED
        assert abi.dn_set_state(layer.handle, 0, good.S, good.ring, good.ring_pos,
                                check=False) == abi.DN_EFAILED
        after = layer.get_state()  # the engine continues from what the card holds
        assert np.array_equal(after.S, good.S)
        assert np.array_equal(after.ring, good.ring)
        assert np.array_equal(after.ring_pos, good.ring_pos)
    finally:
        layer.destroy()


def test_bounded_device_wait_that_runs_out_is_reported():
    """Every wait of the step's kernels is bounded and records a give-up in
    the layer's device error word.  Here one thread waits 2 ms for a flag
    that nothing sets, ahead of a step: the step itself completes as usual
    (its state equals a second layer's that ran the same steps), the next
    get_state still copies the state out but returns DN_ECUDA, and the layer
    is off from then on.  A cancelled request changes nothing."""
    rng = np.random.default_rng(5)
    w = make_weights(TINY, rng)
    layer = GpuLayer.create(TINY, w, 2)
    twin = GpuLayer.create(TINY, w, 2)
    try:
        s1 = WorkloadStream(custom_workload("t", TINY, 2, 8, seed=6))
        s2 = WorkloadStream(custom_workload("t", TINY, 2, 8, seed=6))
        abi.dn_debug_expire_wait(layer.handle, 2000)
        abi.dn_debug_expire_wait(layer.handle, 0)  # cancelled
        _run(layer, s1, 2, 2)
        _run(twin, s2, 3, 2)
        abi.dn_debug_expire_wait(layer.handle, 2000)
        x, gates = s1.next_step()
        xd, gd, bd, od = _dev_inputs(x, *gates[0])
        assert abi.dn_step(layer.handle, 2, xd, gd, bd, od, check=False) == abi.DN_OK
        S = np.empty((2, TINY.n_v_heads, TINY.dk, TINY.dv), np.float32)
        ring = np.empty((2, TINY.conv_k - 1, TINY.conv_ch), np.float32)
        rp = np.empty(2, np.int32)
        assert abi.dn_get_state(layer.handle, 0, 2, S, ring, rp, check=False) == abi.DN_ECUDA
        ref = twin.get_state()
        assert np.array_equal(S, ref.S) and np.array_equal(ring, ref.ring)
        assert np.array_equal(rp, ref.ring_pos)
        assert abi.dn_step(layer.handle, 2, xd, gd, bd, od, check=False) == abi.DN_EFAILED
    finally:
        layer.destroy()
        twin.destroy()


@pytest.mark.parametrize("batch", [1, 16])
def test_zero_gates_leave_the_state_bitwise_unchanged(batch):
    """g = 0 (no decay) and beta = 0 (no write) make the delta rule the
    identity on S: S <- 1 * S + k (0 * (v - S^T k)).  After several steps
    the state equals the initial one bit for bit, on the CUDA-core (batch 1)
    and tensor-core (batch 16) projection paths, while the readouts still
    match the oracle (checked by the parity tests on the same kernels)."""
    torch = _torch()
    wl = custom_workload("zero_gates", SHAPE_35B, batch=batch, steps=3, seed=88, init_std=0.02)
    stream = WorkloadStream(wl)
    s0 = stream.states[0]
    layer = GpuLayer.create(wl.cfg, stream.weights[0], batch, s0)
    try:
        z = torch.zeros((batch, wl.cfg.n_v_heads), device="cuda")
        out = torch.empty((batch, wl.cfg.hidden), device="cuda")
        for _ in range(3):
            x, _ = stream.next_step()
            abi.dn_step(layer.handle, batch, torch.from_numpy(x).cuda(), z, z, out)
        assert np.array_equal(layer.get_state().S, s0.S)
        assert torch.isfinite(out).all()
    finally:
        layer.destroy()


def test_device_memory_accounting_returns_to_zero():
    base = abi.dn_device_bytes()
    w = make_weights(TINY, np.random.default_rng(4))
    for i in range(10):
        layer = GpuLayer.create(TINY, w, 1 + 7 * i)
        assert abi.dn_device_bytes() > base
        layer.destroy()
        assert abi.dn_device_bytes() == base
    assert base == 0


def test_two_runs_are_bitwise_identical():
    wl = custom_workload("det", SHAPE_35B, batch=3, steps=6, seed=9, init_std=0.02)
    outs, states = [], []
    for _ in range(2):
        stream = WorkloadStream(wl)
        layer = GpuLayer.create(wl.cfg, stream.weights[0], 3, stream.states[0])
        try:
            outs.append(_run(layer, stream, 6, 3))
            states.append(layer.get_state())
        finally:
            layer.destroy()
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)
    assert np.array_equal(states[0].S, states[1].S)
    assert np.array_equal(states[0].ring, states[1].ring)


def test_host_pointer_step_equals_device_pointer_step():
    wl = custom_workload("hd", TINY, batch=4, steps=5, seed=10, init_std=0.1)
    s1, s2 = WorkloadStream(wl), WorkloadStream(wl)
    a = GpuLayer.create(TINY, s1.weights[0], 4, s1.states[0])
    b = GpuLayer.create(TINY, s2.weights[0], 4, s2.states[0])
    try:
        for _ in range(5):
            x, gates = s1.next_step()
            s2.next_step()
            out_h = np.empty_like(x)
            abi.dn_step(a.handle, 4, x, gates[0][0], gates[0][1], out_h)  # host pointers
            xd, gd, bd, od = _dev_inputs(x, *gates[0])
            abi.dn_step(b.handle, 4, xd, gd, bd, od)
            assert np.array_equal(out_h, od.cpu().numpy())
        assert np.array_equal(a.get_state().S, b.get_state().S)
    finally:
        a.destroy()
        b.destroy()


def test_sequences_beyond_batch_are_untouched():
    rng = np.random.default_rng(11)
    w = make_weights(TINY, rng)
    st = random_state(TINY, 7, rng, 0.2)
    layer = GpuLayer.create(TINY, w, 7, st)
    try:
        stream = WorkloadStream(custom_workload("u", TINY, 7, 4, seed=12))
        _run(layer, stream, 4, 5)
        back = layer.get_state()
        assert np.array_equal(back.S[5:], st.S[5:])
        assert np.array_equal(back.ring[5:], st.ring[5:])
        assert np.array_equal(back.ring_pos[5:], st.ring_pos[5:])
        assert not np.array_equal(back.S[:5], st.S[:5])
    finally:
        layer.destroy()


def test_checkpoint_resume_is_bitwise():
    """Checkpoint at step 128 with get_state, restore into a fresh layer with
    set_state and continue: identical to 256 uninterrupted steps."""
    wl = custom_workload("ck", SHAPE_35B, batch=2, steps=256, seed=13, init_std=0.02)
    s_full = WorkloadStream(wl)
    full = GpuLayer.create(wl.cfg, s_full.weights[0], 2, s_full.states[0])
    s_ck = WorkloadStream(wl)
    first = GpuLayer.create(wl.cfg, s_ck.weights[0], 2, s_ck.states[0])
    try:
        out_full = _run(full, s_full, 256, 2)
        _run(first, s_ck, 128, 2)
        ck = first.get_state()
        first.destroy()
        second = GpuLayer.create(wl.cfg, s_ck.weights[0], 2, ck)
        try:
            out_rest = _run(second, s_ck, 128, 2)
            assert np.array_equal(out_rest[-1], out_full[-1])
            fs, ss = full.get_state(), second.get_state()
            assert np.array_equal(fs.S, ss.S) and np.array_equal(fs.ring, ss.ring)
            assert np.array_equal(fs.ring_pos, ss.ring_pos)
        finally:
            second.destroy()
    finally:
        full.destroy()
        first.destroy()


def test_two_runs_are_bitwise_identical_on_the_tensor_core_path():
    """Batch 16 of the 35B shape takes the tensor-core projections and the
    persistent state kernel; the stream-K partials are summed in slot order,
    so two runs agree bit for bit."""
    wl = custom_workload("det16", SHAPE_35B, batch=16, steps=4, seed=19, init_std=0.02)
    outs, states = [], []
    for _ in range(2):
        stream = WorkloadStream(wl)
        layer = GpuLayer.create(wl.cfg, stream.weights[0], 16, stream.states[0])
        try:
            assert abi.dn_step_kernels(layer.handle, 16) == 5  # pack, GEMM, state, GEMM, reduce
            outs.append(_run(layer, stream, 4, 16))
            states.append(layer.get_state())
        finally:
            layer.destroy()
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)
    assert np.array_equal(states[0].S, states[1].S)


def test_profiled_step_records_five_stage_events_and_changes_nothing():
    torch = _torch()
    wl = custom_workload("prof", SHAPE_35B, batch=16, steps=2, seed=23, init_std=0.02)
    s1, s2 = WorkloadStream(wl), WorkloadStream(wl)
    a = GpuLayer.create(wl.cfg, s1.weights[0], 16, s1.states[0])
    b = GpuLayer.create(wl.cfg, s2.weights[0], 16, s2.states[0])
    try:
        assert abi.dn_step_kernels(a.handle, 1) == 4
        assert abi.dn_step_kernels(a.handle, 17) == 0
        with pytest.raises(ValueError):
            abi.dn_profile_next_step(a.handle, [torch.cuda.Event(enable_timing=True)] * 4)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        for e in evs:  # torch creates the CUDA event on first record
            e.record()
        abi.dn_profile_next_step(a.handle, evs)
        x, gates = s1.next_step()
        s2.next_step()
        xd, gd, bd, od = _dev_inputs(x, *gates[0])
        abi.dn_step(a.handle, 16, xd, gd, bd, od)
        xd2, gd2, bd2, od2 = _dev_inputs(x, *gates[0])
        abi.dn_step(b.handle, 16, xd2, gd2, bd2, od2)
        torch.cuda.synchronize()
        times = [evs[i].elapsed_time(evs[i + 1]) for i in range(4)]
        assert all(t >= 0.0 for t in times) and sum(times) > 0.0
        assert np.array_equal(od.cpu().numpy(), od2.cpu().numpy())
    finally:
        a.destroy()
        b.destroy()


def test_state_copies_wait_for_steps_on_another_stream():
    """Steps enqueued on a non-blocking stream other than the layer's: an
    immediate dn_get_state (no synchronisation by the caller) already sees
    every one of them, and a dn_set_state issued right after the steps lands
    after them (the next get returns exactly what was set)."""
    torch = _torch()
    wl = custom_workload("xstream_35b_b64", SHAPE_35B, batch=64, steps=24, seed=21, init_std=0.02)
    st = WorkloadStream(wl)
    layer = GpuLayer.create(wl.cfg, st.weights[0], wl.batch, st.states[0])
    try:
        side = torch.cuda.Stream()  # torch pool streams are non-blocking
        steps = []
        for _ in range(24):
            x, gates = st.next_step()
            steps.append(_dev_inputs(x, gates[0][0], gates[0][1]))
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            for xd, gd, bd, od in steps:
                abi.dn_step(layer.handle, wl.batch, xd, gd, bd, od, stream=side.cuda_stream)
        early = layer.get_state()          # no synchronisation before it
        torch.cuda.synchronize()
        late = layer.get_state()
        assert np.array_equal(early.S, late.S)
        assert np.array_equal(early.ring, late.ring)
        assert np.array_equal(early.ring_pos, late.ring_pos)
        # set_state right after more steps on the side stream
        with torch.cuda.stream(side):
            for xd, gd, bd, od in steps[:8]:
                abi.dn_step(layer.handle, wl.batch, xd, gd, bd, od, stream=side.cuda_stream)
        rng = np.random.default_rng(5)
        want = random_state(wl.cfg, wl.batch, rng, 0.01)
        abi.dn_set_state(layer.handle, 0, want.S, want.ring, want.ring_pos)
        torch.cuda.synchronize()
        got = layer.get_state()
        assert np.array_equal(got.S, want.S)
        assert np.array_equal(got.ring, want.ring)
        assert np.array_equal(got.ring_pos, want.ring_pos)
    finally:
        layer.destroy()
