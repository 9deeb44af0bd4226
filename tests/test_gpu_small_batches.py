"""GPU parity of small-batch decode steps (the CUDA-core projections at one
sequence, the tensor-core ones from two) against the float64 oracle on the
same seeded inputs: more (sequence, head) state items than SMs, every conv
width of the streaming state kernel, per-key gates with int4 weights, one
layer stepped at CUDA-core and tensor-core batch sizes in turn, and a
captured CUDA graph of several steps replayed several times."""
import numpy as np
import pytest

from gated_deltanet_hybrid_gb300 import abi
from gated_deltanet_hybrid_gb300.inputs import SHAPE_35B, DNConfig, DNState, WorkloadStream, custom_workload

from harness import REL_TOL, GpuLayer, rel_err, run_parity

pytestmark = pytest.mark.gpu

SMALL_128 = dict(hidden=512, n_qk_heads=2, n_v_heads=4, dk=128, dv=128)


def _assert_ok(w):
    assert w["out"] <= REL_TOL, w
    assert w["S"] <= REL_TOL, w
    assert w["ring"] <= REL_TOL, w
    assert w["ring_pos_equal"], w


def test_35b_batch7_more_state_items_than_sms():
    """7 x 32 = 224 (sequence, head) items on 152 SMs."""
    wl = custom_workload("35b_b7", SHAPE_35B, batch=7, steps=12, seed=707, init_std=0.02)
    _assert_ok(run_parity(wl, sample=np.array([0, 3, 6])))


@pytest.mark.parametrize("conv_k", [2, 3, 4])
@pytest.mark.parametrize("batch", [1, 2, 5])
def test_conv_widths(conv_k, batch):
    cfg = DNConfig(**SMALL_128, conv_k=conv_k)
    wl = custom_workload("small_conv", cfg, batch=batch, steps=20, seed=60 + 7 * conv_k + batch, init_std=0.05)
    _assert_ok(run_parity(wl))


@pytest.mark.parametrize("batch", [1, 6])
def test_key_gate_with_int4_weights(batch):
    cfg = DNConfig(**SMALL_128, key_gate=True, int4=True)
    wl = custom_workload("small_kg_i4", cfg, batch=batch, steps=20, seed=90 + batch, init_std=0.05)
    _assert_ok(run_parity(wl))


def _oracle_layers(cfg, w, s0, n):
    from oracle import OracleLayer
    return [OracleLayer(cfg, w, DNState(s0.S[i:i + 1], s0.ring[i:i + 1], s0.ring_pos[i:i + 1]))
            for i in range(n)]


def test_cuda_core_and_tensor_core_batches_on_one_layer():
    """Steps of 1 sequence (CUDA-core projections) and of 3 and 9 (tensor-core
    projections) on one layer, in turn: all read and advance the same state,
    ring and ring positions."""
    import torch
    cfg = DNConfig(**SMALL_128)
    wl = custom_workload("mixed", cfg, batch=9, steps=12, seed=3309, init_std=0.05)
    st = WorkloadStream(wl)
    w, s0 = st.weights[0], st.states[0]
    gpu = GpuLayer.create(cfg, w, 9, s0)
    ora = _oracle_layers(cfg, w, s0, 9)
    dev = torch.device("cuda")
    try:
        assert abi.dn_step_kernels(gpu.handle, 1) == 4
        assert abi.dn_step_kernels(gpu.handle, 3) == 5
        worst = 0.0
        for t in range(wl.steps):
            x, gates = st.next_step()
            g, beta = gates[0]
            B = (1, 3, 9)[t % 3]
            x_d = torch.from_numpy(np.ascontiguousarray(x[:B])).to(dev)
            g_d = torch.from_numpy(np.ascontiguousarray(g[:B])).to(dev)
            b_d = torch.from_numpy(np.ascontiguousarray(beta[:B])).to(dev)
            out_d = torch.empty_like(x_d)
            abi.dn_step(gpu.handle, B, x_d, g_d, b_d, out_d)
            got = out_d.cpu().numpy()
            for i in range(B):
                ref = ora[i].step(x[i:i + 1], g[i:i + 1], beta[i:i + 1])
                worst = max(worst, rel_err(got[i:i + 1], ref))
        assert worst <= REL_TOL, worst
        gs = gpu.get_state()
        for i in range(9):
            assert rel_err(gs.S[i:i + 1], ora[i].S) <= REL_TOL, i
            assert rel_err(gs.ring[i:i + 1], ora[i].ring) <= REL_TOL, i
            assert np.array_equal(gs.ring_pos[i:i + 1], ora[i].ring_pos), i
    finally:
        gpu.destroy()


def test_graph_replays():
    """Four steps captured in one CUDA graph and replayed three times give the
    oracle's twelve steps (every input buffer is refilled between replays)."""
    import torch
    from oracle import OracleLayer
    cfg = DNConfig(**SMALL_128)
    B, per, reps = 2, 4, 3
    wl = custom_workload("graph", cfg, batch=B, steps=1 + per * reps, seed=4404, init_std=0.05)
    st = WorkloadStream(wl)
    w, s0 = st.weights[0], st.states[0]
    gpu = GpuLayer.create(cfg, w, B, s0)
    ora = OracleLayer(cfg, w, DNState(s0.S, s0.ring, s0.ring_pos))
    dev = torch.device("cuda")
    xs = torch.empty((per, B, cfg.hidden), dtype=torch.float32, device=dev)
    gs = torch.empty((per, B, cfg.n_v_heads), dtype=torch.float32, device=dev)
    bs = torch.empty((per, B, cfg.n_v_heads), dtype=torch.float32, device=dev)
    outs = torch.empty_like(xs)
    worst = 0.0
    try:
        # one eager step first (also sets the kernels' launch attributes)
        x, ((g, beta),) = st.next_step()
        xs[0].copy_(torch.from_numpy(x))
        gs[0].copy_(torch.from_numpy(g))
        bs[0].copy_(torch.from_numpy(beta))
        abi.dn_step(gpu.handle, B, xs[0], gs[0], bs[0], outs[0])
        worst = max(worst, rel_err(outs[0].cpu().numpy(), ora.step(x, g, beta)))
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        torch.cuda.synchronize()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(graph, stream=cap):
                for i in range(per):
                    abi.dn_step(gpu.handle, B, xs[i], gs[i], bs[i], outs[i])
        torch.cuda.synchronize()
        for _ in range(reps):
            refs = []
            for i in range(per):
                x, ((g, beta),) = st.next_step()
                xs[i].copy_(torch.from_numpy(x))
                gs[i].copy_(torch.from_numpy(g))
                bs[i].copy_(torch.from_numpy(beta))
                refs.append(ora.step(x, g, beta))
            graph.replay()
            torch.cuda.synchronize()
            for i in range(per):
                worst = max(worst, rel_err(outs[i].cpu().numpy(), refs[i]))
        assert worst <= REL_TOL, worst
        s = gpu.get_state()
        assert rel_err(s.S, ora.S) <= REL_TOL
        assert rel_err(s.ring, ora.ring) <= REL_TOL
        assert np.array_equal(s.ring_pos, ora.ring_pos)
    finally:
        gpu.destroy()
