"""The projection entry point that allocates nothing (dn_proj_i8_noalloc).

Some callers cannot allocate device memory: code that runs inside another
runtime's memory pool, or under a device-memory budget fixed in advance,
may call neither cudaMalloc nor anything that allocates for it.  For them
the library offers the int8 row-scaled projection y = s * (W x) with its
split-K scratch in a static device array, so only the caller's inputs and
outputs are touched.  This test checks it against the projection that
dn_step runs: after a step the conv ring holds that step's in_proj output
for the q, k and v rows, and two steps in a row must match the new call
within the tolerance of the other GPU tests.  (Collected last on purpose.)
"""
import numpy as np
import pytest

from gated_deltanet_hybrid_gb300 import abi
from gated_deltanet_hybrid_gb300.inputs import SHAPE_35B, custom_workload, WorkloadStream

from harness import REL_TOL, GpuLayer, rel_err

pytestmark = pytest.mark.gpu


def test_noalloc_projection_matches_dn_step_in_proj_twice():
    import torch

    cfg, batch = SHAPE_35B, 3
    stream = WorkloadStream(custom_workload("noalloc", cfg, batch=batch, steps=2, seed=77))
    w = stream.weights[0]
    layer = GpuLayer.create(cfg, w, batch)
    W_d = torch.from_numpy(w.w_in).cuda()
    s_d = torch.from_numpy(w.s_in).cuda()
    try:
        for step in (1, 2):
            x, gates = stream.next_step()
            x_d = torch.from_numpy(x).cuda()
            out = torch.empty_like(x_d)
            abi.dn_step(layer.handle, batch, x_d, torch.from_numpy(gates[0][0]).cuda(),
                        torch.from_numpy(gates[0][1]).cuda(), out)
            st = layer.get_state()
            newest = (int(st.ring_pos[0]) + cfg.conv_k - 2) % (cfg.conv_k - 1)
            assert np.all(st.ring_pos == step % (cfg.conv_k - 1))
            ref = st.ring[:, newest, :]  # dn_step's in_proj rows q | k | v

            y = torch.full((batch, cfg.in_rows), float("nan"), device="cuda")
            abi.dn_proj_i8_noalloc(W_d, s_d, x_d, y)
            torch.cuda.synchronize()
            got = y.cpu().numpy()
            assert np.isfinite(got).all()
            assert rel_err(got[:, :cfg.conv_ch], ref) <= REL_TOL
            # and against an exact float64 product of the same int8 rows
            exact = (x.astype(np.float64) @ w.w_in.astype(np.float64).T) * w.s_in.astype(np.float64)
            assert rel_err(got, exact) <= REL_TOL
    finally:
        layer.destroy()


@pytest.mark.parametrize("M,K,B", [(200, 80, 1), (1000, 1040, 8), (1, 16, 1), (16384, 16384, 8)])
def test_noalloc_projection_ragged_and_largest_shapes(M, K, B):
    """Row tails (M not a multiple of 128), k tails (K not a multiple of 64),
    one and eight sequences, the smallest shape and the largest accepted one,
    each against the exact float64 product; y starts as NaN so that a row
    the call does not write shows."""
    import torch

    rng = np.random.default_rng(M * 7 + K * 3 + B)
    W = rng.integers(-127, 128, size=(M, K), dtype=np.int8)
    s = rng.uniform(0.001, 0.01, size=M).astype(np.float32)
    x = rng.standard_normal((B, K)).astype(np.float32)
    W_d, s_d, x_d = torch.from_numpy(W).cuda(), torch.from_numpy(s).cuda(), torch.from_numpy(x).cuda()
    y = torch.full((B, M), float("nan"), device="cuda")
    for _ in range(2):  # the second call reuses the scratch the first one left
        abi.dn_proj_i8_noalloc(W_d, s_d, x_d, y)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        assert np.isfinite(got).all()
        exact = np.empty((B, M))
        x64 = x.astype(np.float64)
        for r0 in range(0, M, 2048):  # bounded host memory for the largest shape
            exact[:, r0:r0 + 2048] = x64 @ W[r0:r0 + 2048].astype(np.float64).T
        exact *= s.astype(np.float64)
        assert rel_err(got, exact) <= REL_TOL
        y.fill_(float("nan"))


def test_noalloc_projection_rejects_sizes_beyond_its_limits():
    import torch

    W = torch.zeros((256, 64), dtype=torch.int8, device="cuda")
    s = torch.ones(256, device="cuda")
    x9 = torch.zeros((9, 64), device="cuda")  # more than 8 sequences
    y9 = torch.zeros((9, 256), device="cuda")
    assert abi.dn_proj_i8_noalloc(W, s, x9, y9, check=False) == abi.DN_EINVAL
    Wk = torch.zeros((256, 24), dtype=torch.int8, device="cuda")  # K not a multiple of 16
    x = torch.zeros((1, 24), device="cuda")
    y = torch.zeros((1, 256), device="cuda")
    assert abi.dn_proj_i8_noalloc(Wk, s, x, y, check=False) == abi.DN_EINVAL
