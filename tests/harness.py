"""Shared helpers of the GPU tests: drive a workload through the C ABI and the
CPU oracle on the same seeded inputs and compare them."""
from __future__ import annotations

import dataclasses

import numpy as np

from gated_deltanet_hybrid_gb300 import abi
from gated_deltanet_hybrid_gb300.inputs import DNState, Workload, WorkloadStream

#: max |gpu - ref| / max |ref| per tensor and checkpoint (fp32 state and
#: accumulation against the float64 oracle)
REL_TOL = 2e-3


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.abs(ref).max()
    if scale == 0.0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / scale)


def elementwise_rel(got: np.ndarray, ref: np.ndarray, floor: float = 1e-3) -> float:
    """Element-wise relative error with a floor of floor * max|ref|."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.maximum(np.abs(ref), floor * np.abs(ref).max())
    den[den == 0] = 1.0
    return float((np.abs(got - ref) / den).max())


@dataclasses.dataclass
class GpuLayer:
    """A layer created through the ABI, with device buffers for one step."""

    handle: object
    cfg: object
    max_batch: int

    @classmethod
    def create(cls, cfg, weights, max_batch: int, state: DNState | None = None):
        h = abi.dn_create(cfg, weights, max_batch)
        layer = cls(h, cfg, max_batch)
        if state is not None:
            abi.dn_set_state(h, 0, np.ascontiguousarray(state.S), np.ascontiguousarray(state.ring),
                             np.ascontiguousarray(state.ring_pos))
        return layer

    def get_state(self, seq0: int = 0, n: int | None = None) -> DNState:
        c = self.cfg
        n = self.max_batch - seq0 if n is None else n
        S = np.empty((n, c.n_v_heads, c.dk, c.dv), np.float32)
        ring = np.empty((n, c.conv_k - 1, c.conv_ch), np.float32)
        rp = np.empty(n, np.int32)
        abi.dn_get_state(self.handle, seq0, n, S, ring, rp)
        return DNState(S, ring, rp)

    def get_seqs(self, seqs) -> DNState:
        parts = [self.get_state(int(s), 1) for s in seqs]
        return DNState(np.concatenate([p.S for p in parts]), np.concatenate([p.ring for p in parts]),
                       np.concatenate([p.ring_pos for p in parts]))

    def destroy(self):
        if self.handle is not None:
            abi.dn_destroy(self.handle)
            self.handle = None


def run_parity(wl: Workload, steps: int | None = None, sample=None, checkpoints=None,
               max_batch: int | None = None):
    """Run a single-layer workload on the GPU (all sequences) and in the
    oracle (the sampled sequences) and return the worst errors seen.

    Returns dict with keys out (max over steps), S, ring (max over
    checkpoints), ring_pos_equal (bool), elementwise (max over all)."""
    import torch
    from oracle import OracleLayer

    steps = wl.steps if steps is None else steps
    checkpoints = tuple(c for c in (checkpoints or wl.checkpoints or (steps,)) if c <= steps)
    if steps not in checkpoints:
        checkpoints = checkpoints + (steps,)
    B = wl.batch
    sample = np.arange(B) if sample is None else np.asarray(sample)
    st = WorkloadStream(wl)
    w, s0 = st.weights[0], st.states[0]
    gpu = GpuLayer.create(wl.cfg, w, max_batch or B, s0 if wl.init_std > 0 else None)
    ora = OracleLayer(wl.cfg, w, DNState(s0.S[sample], s0.ring[sample], s0.ring_pos[sample]))
    dev = torch.device("cuda")
    x_d = torch.empty((B, wl.cfg.hidden), dtype=torch.float32, device=dev)
    gshape = (B, wl.cfg.n_v_heads, wl.cfg.dk) if getattr(wl.cfg, "key_gate", False) else (B, wl.cfg.n_v_heads)
    g_d = torch.empty(gshape, dtype=torch.float32, device=dev)
    b_d = torch.empty((B, wl.cfg.n_v_heads), dtype=torch.float32, device=dev)
    out_d = torch.empty_like(x_d)
    worst = {"out": 0.0, "S": 0.0, "ring": 0.0, "elementwise_out": 0.0, "ring_pos_equal": True}
    try:
        for t in range(1, steps + 1):
            x, gates = st.next_step()
            g, beta = gates[0]
            x_d.copy_(torch.from_numpy(x))
            if g is None:  # device gates
                abi.dn_step(gpu.handle, B, x_d, None, None, out_d)
                ref = ora.step(x[sample])
            else:
                g_d.copy_(torch.from_numpy(g))
                b_d.copy_(torch.from_numpy(beta))
                abi.dn_step(gpu.handle, B, x_d, g_d, b_d, out_d)
                ref = ora.step(x[sample], g[sample], beta[sample])
            got = out_d.cpu().numpy()[sample]
            worst["out"] = max(worst["out"], rel_err(got, ref))
            worst["elementwise_out"] = max(worst["elementwise_out"], elementwise_rel(got, ref))
            if t in checkpoints:
                gs = gpu.get_seqs(sample)
                worst["S"] = max(worst["S"], rel_err(gs.S, ora.S))
                worst["ring"] = max(worst["ring"], rel_err(gs.ring, ora.ring))
                worst["ring_pos_equal"] &= bool(np.array_equal(gs.ring_pos, ora.ring_pos))
    finally:
        gpu.destroy()
    return worst


def run_prefill_parity(wl: Workload, n_tokens: int, sample=None, max_batch: int | None = None,
                       decode_after: int = 0):
    """A prompt of n_tokens tokens through dn_prefill (all sequences) and
    through the oracle token by token (the sampled sequences), then
    `decode_after` dn_step calls on both; returns the worst errors of the
    outputs (every token), and of S and the ring at the end, and whether the
    ring positions match."""
    import torch
    from oracle import OracleLayer, prefill

    B = wl.batch
    sample = np.arange(B) if sample is None else np.asarray(sample)
    st = WorkloadStream(wl)
    w, s0 = st.weights[0], st.states[0]
    gpu = GpuLayer.create(wl.cfg, w, max_batch or B, s0 if wl.init_std > 0 else None)
    ora = OracleLayer(wl.cfg, w, DNState(s0.S[sample], s0.ring[sample], s0.ring_pos[sample]))
    steps = [st.next_step() for _ in range(n_tokens)]
    x = np.stack([s_[0] for s_ in steps], axis=1)                       # [B][S][hidden]
    dev = getattr(wl.cfg, "device_gates", False)
    g = None if dev else np.stack([s_[1][0][0] for s_ in steps], axis=1)
    beta = None if dev else np.stack([s_[1][0][1] for s_ in steps], axis=1)
    worst = {"out": 0.0, "S": 0.0, "ring": 0.0, "ring_pos_equal": True}
    try:
        cuda = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
        out_d = torch.empty((B, n_tokens, wl.cfg.hidden), dtype=torch.float32, device="cuda")
        abi.dn_prefill(gpu.handle, B, n_tokens, cuda(x), cuda(g), cuda(beta), out_d)
        ref = prefill(ora, x[sample], None if g is None else g[sample], None if beta is None else beta[sample])
        got = out_d.cpu().numpy()[sample]
        for t in range(n_tokens):
            worst["out"] = max(worst["out"], rel_err(got[:, t], ref[:, t]))
        for _ in range(decode_after):
            xs, gates = st.next_step()
            gs, bs = gates[0]
            o = torch.empty((B, wl.cfg.hidden), dtype=torch.float32, device="cuda")
            abi.dn_step(gpu.handle, B, cuda(xs), cuda(gs), cuda(bs), o)
            r = ora.step(xs[sample], None if gs is None else gs[sample], None if bs is None else bs[sample])
            worst["out"] = max(worst["out"], rel_err(o.cpu().numpy()[sample], r))
        gs_ = gpu.get_seqs(sample)
        worst["S"] = rel_err(gs_.S, ora.S)
        worst["ring"] = rel_err(gs_.ring, ora.ring)
        worst["ring_pos_equal"] = bool(np.array_equal(gs_.ring_pos, ora.ring_pos))
    finally:
        gpu.destroy()
    return worst
