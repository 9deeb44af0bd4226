"""The 30-layer stack (the pages' model runs 30 DeltaNet layers per token;
page "qwen36: run the DeltaNet layer end to end on the card (Q36_DN_GPU=1)",
section "Measured"): 49 prompt tokens token-serially, then 200 decode
tokens, batch 1 and 16, through dn_stack_step (pre-norm, layer, residual add
per layer) against the oracle's stack_step on sampled sequences."""
import numpy as np
import pytest

from gated_deltanet_hybrid_gb300 import abi
from gated_deltanet_hybrid_gb300.inputs import WORKLOADS, WorkloadStream, zero_state

from harness import REL_TOL, GpuLayer, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,sample", [("stack30_b1", [0]), ("stack30_b16", [0, 15])])
def test_stack30_matches_oracle(name, sample):
    import torch
    from oracle import OracleLayer, stack_step

    wl = WORKLOADS[name]
    cfg, B, L = wl.cfg, wl.batch, wl.layers
    sample = np.asarray(sample)
    st = WorkloadStream(wl)
    layers = [GpuLayer.create(cfg, w, B) for w in st.weights]
    oracles = [OracleLayer(cfg, w, zero_state(cfg, len(sample))) for w in st.weights]
    handles = [l.handle for l in layers]
    h = torch.empty((B, cfg.hidden), dtype=torch.float32, device="cuda")
    g_d = torch.empty((L, B, cfg.n_v_heads), dtype=torch.float32, device="cuda")
    b_d = torch.empty_like(g_d)
    worst = 0.0
    try:
        for _ in range(wl.prompt + wl.steps):
            x, gates = st.next_step()
            h.copy_(torch.from_numpy(x))
            g_d.copy_(torch.from_numpy(np.stack([g for g, _ in gates])))
            b_d.copy_(torch.from_numpy(np.stack([b for _, b in gates])))
            abi.dn_stack_step(handles, B, h, g_d, b_d)
            ref = stack_step(oracles, x[sample], [(g[sample], b[sample]) for g, b in gates])
            worst = max(worst, rel_err(h.cpu().numpy()[sample], ref))
        assert worst <= REL_TOL, worst
        for l in (0, L - 1):  # the first and the last layer's state
            got, ora = layers[l].get_seqs(sample), oracles[l]
            assert rel_err(got.S, ora.S) <= REL_TOL
            assert rel_err(got.ring, ora.ring) <= REL_TOL
            assert np.array_equal(got.ring_pos, ora.ring_pos)
    finally:
        for l in layers:
            l.destroy()


def test_stack_step_rejects_bad_arguments():
    import torch
    from gated_deltanet_hybrid_gb300.inputs import TINY, make_weights

    w = make_weights(TINY, np.random.default_rng(3))
    a = GpuLayer.create(TINY, w, 2)
    try:
        h = torch.zeros((4, TINY.hidden), device="cuda")
        g = torch.zeros((1, 4, TINY.n_v_heads), device="cuda")
        assert abi.dn_stack_step([a.handle], 4, h, g, g, check=False) == abi.DN_EINVAL  # batch > max_batch
        assert abi.dn_stack_step([a.handle], 1, h, g, g, eps=-1.0, check=False) == abi.DN_EINVAL
        with pytest.raises(TypeError):
            abi.dn_stack_step([a.handle], 1, h.cpu(), g, g)
    finally:
        a.destroy()
