"""Seeded synthetic inputs for the gated-DeltaNet decode step.

This module only draws random numbers and lays them out.  It holds none of
the step's arithmetic, and both sides of a parity check (the CUDA path and
the CPU oracle) read the very same arrays produced here.

The workloads follow the shapes of the 35B hybrid model named on the page
"qwen36: run the DeltaNet layer end to end on the card (Q36_DN_GPU=1)"
(section "Measured": 30 DeltaNet layers, a 49-token prompt, 200 decoded
tokens) and the weight format of "feat(qwen36): the dense trunk places
itself" (section "What this adds", item 1: int8 rows with one fp32 scale
each, in_proj fused as qkv ++ z).

Draw order, with ``numpy.random.Generator(PCG64(seed))``:
  1. weights: W_in, s_in, w_conv, w_norm, W_out, s_out
  2. initial state (only when the workload asks for a random one): S, ring
  3. per decode step, in step order: x, then the two gate draws.

The gates travel as inputs (the page computes the two small a/b gate
projections on the host and hands their values to the kernels).  The
workload turns its two normal draws a, b into the per-head log-decay g and
write strength beta with g = -0.5 * softplus(a) and beta = sigmoid(b), in
float64, then rounds both to float32 once; every consumer reads those
float32 values.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Iterator

import numpy as np


@dataclasses.dataclass(frozen=True)
class DNConfig:
    """Dimensions of one gated-DeltaNet layer and its two epsilons."""

    hidden: int
    n_qk_heads: int
    n_v_heads: int
    dk: int
    dv: int
    conv_k: int = 4
    l2_eps: float = 1e-6
    norm_eps: float = 1e-6
    q_scale: float | None = None  # None: 1/sqrt(dk)
    key_gate: bool = False        # per-key-channel decay: g is [n_v_heads][dk] per sequence
    device_gates: bool = False    # the a/b gate projections are int8 rows of the layer (no host gates)
    int4: bool = False            # projection weights are per-row int4 (integers in [-8, 7]) instead of int8

    @property
    def gate_width(self) -> int:
        """Log-decay values per head and step: dk with the per-key gate, else 1."""
        return self.dk if self.key_gate else 1

    @property
    def qscale(self) -> float:
        return 1.0 / math.sqrt(self.dk) if self.q_scale is None else float(self.q_scale)

    @property
    def qk_dim(self) -> int:
        return self.n_qk_heads * self.dk

    @property
    def v_dim(self) -> int:
        return self.n_v_heads * self.dv

    @property
    def conv_ch(self) -> int:
        return 2 * self.qk_dim + self.v_dim

    @property
    def in_rows(self) -> int:
        return self.conv_ch + self.v_dim

    @property
    def gate_rows(self) -> int:
        """Rows of the a/b gate projections: n_v_heads * gate_width for a,
        n_v_heads for b (0 when the gates come from the caller)."""
        return self.n_v_heads * (self.gate_width + 1) if self.device_gates else 0


TINY = DNConfig(hidden=256, n_qk_heads=2, n_v_heads=4, dk=32, dv=32)
SHAPE_35B = DNConfig(hidden=2048, n_qk_heads=16, n_v_heads=32, dk=128, dv=128)


@dataclasses.dataclass
class DNWeights:
    w_in: np.ndarray    # int8  [in_rows][hidden]  rows: q | k | v | z
    s_in: np.ndarray    # f32   [in_rows]
    w_conv: np.ndarray  # f32   [conv_ch][conv_k]  tap conv_k-1 meets the newest input
    w_norm: np.ndarray  # f32   [dv]
    w_out: np.ndarray   # int8  [hidden][v_dim]
    s_out: np.ndarray   # f32   [hidden]
    # device gates only: the a rows (n_v_heads * gate_width) then the b rows
    # (n_v_heads) of the gate projections, their row scales, and the decay
    # coefficient A of each head (g = -A * softplus(a), beta = sigmoid(b))
    w_ab: np.ndarray | None = None     # int8 [gate_rows][hidden]
    s_ab: np.ndarray | None = None     # f32  [gate_rows]
    gate_A: np.ndarray | None = None   # f32  [n_v_heads]


@dataclasses.dataclass
class DNState:
    S: np.ndarray         # f32 [B][n_v_heads][dk][dv]
    ring: np.ndarray      # f32 [B][conv_k-1][conv_ch]
    ring_pos: np.ndarray  # int32 [B]: slot holding the oldest input


def make_weights(cfg: DNConfig, rng: np.random.Generator) -> DNWeights:
    # int4 layers: integers in [-8, 7] (held in int8 arrays) with scales 16x
    # larger, so that the projections' outputs have the int8 layers' size
    lo, hi, sm = (-8, 8, 16.0) if cfg.int4 else (-127, 128, 1.0)
    w_in = rng.integers(lo, hi, size=(cfg.in_rows, cfg.hidden), dtype=np.int8)
    s_in = (rng.uniform(0.001, 0.01, size=cfg.in_rows) * sm).astype(np.float32)
    w_conv = rng.uniform(-0.5, 0.5, size=(cfg.conv_ch, cfg.conv_k)).astype(np.float32)
    w_norm = rng.uniform(0.5, 1.5, size=cfg.dv).astype(np.float32)
    w_out = rng.integers(lo, hi, size=(cfg.hidden, cfg.v_dim), dtype=np.int8)
    s_out = (rng.uniform(0.001, 0.01, size=cfg.hidden) * sm).astype(np.float32)
    w = DNWeights(w_in, s_in, w_conv, w_norm, w_out, s_out)
    if cfg.device_gates:
        # drawn last, so layers without device gates keep their draws; the row
        # scales put a and b near N(0, 1) for x ~ N(0, 1) (int8 uniform in
        # [-127, 127] has standard deviation 73.3), as the configs' a, b are;
        # A = 0.5, the configs' coefficient
        w.w_ab = rng.integers(lo, hi, size=(cfg.gate_rows, cfg.hidden), dtype=np.int8)
        sd = 4.61 if cfg.int4 else 73.3  # standard deviation of the uniform integers
        w.s_ab = (rng.uniform(0.5, 1.5, size=cfg.gate_rows) / (sd * math.sqrt(cfg.hidden))).astype(np.float32)
        w.gate_A = np.full(cfg.n_v_heads, 0.5, np.float32)
    return w


def zero_state(cfg: DNConfig, batch: int) -> DNState:
    return DNState(
        S=np.zeros((batch, cfg.n_v_heads, cfg.dk, cfg.dv), np.float32),
        ring=np.zeros((batch, cfg.conv_k - 1, cfg.conv_ch), np.float32),
        ring_pos=np.zeros(batch, np.int32),
    )


def random_state(cfg: DNConfig, batch: int, rng: np.random.Generator, std: float) -> DNState:
    S = (rng.standard_normal((batch, cfg.n_v_heads, cfg.dk, cfg.dv)) * std).astype(np.float32)
    ring = (rng.standard_normal((batch, cfg.conv_k - 1, cfg.conv_ch)) * std).astype(np.float32)
    return DNState(S=S, ring=ring, ring_pos=np.zeros(batch, np.int32))


def gates_from_ab(a: np.ndarray, b: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """The workload's gate recipe: g = -0.5*softplus(a), beta = sigmoid(b)."""
    a = a.astype(np.float64)
    b = b.astype(np.float64)
    softplus = np.maximum(a, 0.0) + np.log1p(np.exp(-np.abs(a)))
    g = -0.5 * softplus
    beta = 1.0 / (1.0 + np.exp(-b))
    return g.astype(np.float32), beta.astype(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: layer shape, batch, steps, seed and recipe."""

    name: str
    cfg: DNConfig
    batch: int
    steps: int
    seed: int
    init_std: float = 0.0          # 0: zero initial state
    gate: str = "softplus"         # "softplus": a,b ~ N(0,1); "decay_band": exp(g) ~ U(0.9, 1)
    layers: int = 1
    layer_seed0: int | None = None  # per-layer weight seeds (layer_seed0 + l) for stacks
    prompt: int = 0                # stacks: prompt tokens processed token-serially first
    checkpoints: tuple[int, ...] = ()


WORKLOADS = {
    "tiny": Workload("tiny", TINY, batch=1, steps=64, seed=0, checkpoints=(64,)),
    "35b_b1": Workload("35b_b1", SHAPE_35B, batch=1, steps=256, seed=1, checkpoints=(64, 256)),
    "35b_b64": Workload("35b_b64", SHAPE_35B, batch=64, steps=256, seed=2, init_std=0.02,
                        checkpoints=(64, 256)),
    "stack30_b1": Workload("stack30_b1", SHAPE_35B, batch=1, steps=200, seed=3, layers=30,
                           layer_seed0=1000, prompt=49),
    "stack30_b16": Workload("stack30_b16", SHAPE_35B, batch=16, steps=200, seed=3, layers=30,
                            layer_seed0=1000, prompt=49),
    "long_prompt_b8": Workload("long_prompt_b8", SHAPE_35B, batch=8, steps=2048, seed=4,
                               gate="decay_band", checkpoints=(512, 1024, 2048)),
}


class WorkloadStream:
    """Draws a workload's weights, initial state and per-step inputs in order.

    For a single-layer workload the weights come from the workload's own
    generator; a stack draws layer l's weights from PCG64(layer_seed0 + l)
    and keeps the workload's generator for the initial state and the steps.
    """

    def __init__(self, wl: Workload):
        self.wl = wl
        self.rng = np.random.Generator(np.random.PCG64(wl.seed))
        if wl.layers == 1:
            self.weights = [make_weights(wl.cfg, self.rng)]
        else:
            self.weights = [
                make_weights(wl.cfg, np.random.Generator(np.random.PCG64(wl.layer_seed0 + l)))
                for l in range(wl.layers)
            ]
        if wl.init_std > 0.0:
            self.states = [random_state(wl.cfg, wl.batch, self.rng, wl.init_std) for _ in range(wl.layers)]
        else:
            self.states = [zero_state(wl.cfg, wl.batch) for _ in range(wl.layers)]

    def next_step(self) -> tuple[np.ndarray, list[tuple[np.ndarray, np.ndarray]]]:
        """x [B][hidden] f32 and, per layer, (g, beta): g [B][n_v_heads] f32
        ([B][n_v_heads][dk] with the per-key gate), beta [B][n_v_heads] f32;
        (None, None) for a layer with device gates."""
        cfg, B = self.wl.cfg, self.wl.batch
        x = self.rng.standard_normal((B, cfg.hidden)).astype(np.float32)
        gates = []
        gshape = (B, cfg.n_v_heads, cfg.dk) if cfg.key_gate else (B, cfg.n_v_heads)
        for _ in range(self.wl.layers):
            if cfg.device_gates:  # the layer computes its gates from x
                gates.append((None, None))
            elif self.wl.gate == "softplus":
                a = self.rng.standard_normal(gshape)
                b = self.rng.standard_normal((B, cfg.n_v_heads))
                g, _ = gates_from_ab(a, a)
                _, beta = gates_from_ab(b, b)
                gates.append((g, beta))
            elif self.wl.gate == "decay_band":
                u = self.rng.uniform(0.9, 1.0, size=gshape)
                b = self.rng.standard_normal((B, cfg.n_v_heads))
                g = np.log(u).astype(np.float32)
                beta = (1.0 / (1.0 + np.exp(-b))).astype(np.float32)
                gates.append((g, beta))
            else:
                raise ValueError(f"unknown gate recipe {self.wl.gate!r}")
        return x, gates

    def steps(self, n: int) -> Iterator[tuple[np.ndarray, list[tuple[np.ndarray, np.ndarray]]]]:
        for _ in range(n):
            yield self.next_step()


def custom_workload(name: str, cfg: DNConfig, batch: int, steps: int, seed: int,
                    init_std: float = 0.0, gate: str = "softplus") -> Workload:
    """A single-layer workload with other sizes (tests sweep ragged batches)."""
    return Workload(name, cfg, batch=batch, steps=steps, seed=seed, init_std=init_std, gate=gate)
