"""CPU oracle for the gated-DeltaNet decode step (float64, plain numpy).

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import this module.  It shares no code with
the CUDA path: it never imports the product package, and the product never
imports it.  Both read the same seeded input arrays.

What it computes follows the page "qwen36: run the DeltaNet layer end to end
on the card (Q36_DN_GPU=1)", section "What the PR does": in_proj GEMV, causal
conv + SiLU with the ring advancing, per value head the L2 norms of q and k
(double, eps inside the square root), the decay, the delta against the
decayed state, the write-back, out = q^T S over the updated state, the gated
RMSNorm with silu(z), and the out_proj GEMV.  Each function below is one of
those steps, written as its plain definition in float64, in that order.
The fused in_proj (qkv ++ z in one int8 matrix with one fp32 scale per
output row) is from "feat(qwen36): the dense trunk places itself", section
"What this adds", item 1.

Readings where the pages leave a step open (each also listed in the design
notes):
  * int8 row y[o] = s[o] * sum_i W[o, i] x[i]: the scale multiplies the dot
    product of the integer row with x.
  * in_proj rows are [q | k | v | z]; q and k hold n_qk_heads heads of dk,
    v and z hold n_v_heads heads of dv; head h is the contiguous slice
    h*d .. (h+1)*d of its block.
  * value head h reads q/k head h // (n_v_heads // n_qk_heads).
  * the conv is depthwise and causal over the q|k|v channels only, no bias;
    tap conv_k-1 meets the current input; the ring keeps the last conv_k-1
    inputs per channel and ring_pos is the slot of the oldest one.
  * L2 norm: x / sqrt(sum x^2 + l2_eps); q is then multiplied by q_scale.
  * gated RMSNorm over one head's dv values, one weight vector shared by all
    heads: o / sqrt(mean(o^2) + norm_eps) * w_norm * silu(z).
  * the per-key-channel gate of the page's KDA engines (the page says only
    that their gate differs): one log-decay per key index, scaling row i of
    S (S <- diag(exp(g)) S), everything else unchanged.

State S[h] is dk x dv (row i = key index, column j = value index), so the
readout is o[j] = sum_i S[i, j] q[i].
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def silu(x: np.ndarray) -> np.ndarray:
    """silu(x) = x * sigmoid(x) = x / (1 + e^-x)."""
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def softplus(x: np.ndarray) -> np.ndarray:
    """softplus(x) = log(1 + e^x), as max(x, 0) + log1p(e^-|x|) (no overflow)."""
    x = np.asarray(x, F64)
    return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))


def sigmoid(x: np.ndarray) -> np.ndarray:
    """sigmoid(x) = 1 / (1 + e^-x)."""
    x = np.asarray(x, F64)
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-x))


def gate_transform(a: np.ndarray, b: np.ndarray, A: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """The gates from the a/b projections: log-decay g = -A * softplus(a) and
    write strength beta = sigmoid(b), A one coefficient per head (the
    workloads' recipe, g = -softplus(a) * 0.5, beta = sigmoid(b), with A =
    0.5).  a is [..., heads] or [..., heads, dk] (per-key gate), b [..., heads]."""
    a = np.asarray(a, F64)
    A = np.asarray(A, F64)
    g = -(A[:, None] if a.ndim == np.ndim(b) + 1 else A) * softplus(a)
    return g, sigmoid(b)


def int8_rowscaled_gemv(w: np.ndarray, s: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y[..., o] = s[o] * sum_i w[o, i] * x[..., i], in float64.

    One int8 matrix row per output, one fp32 scale per row ("dense-i8"
    entries, "feat(qwen36): the dense trunk places itself", section "What
    this adds").  x may carry leading batch axes; every batch row is the same
    matrix-vector product.
    """
    wf = w.astype(F64, copy=False)
    return (np.asarray(x, F64) @ wf.T) * s.astype(F64)


def causal_conv_silu_step(w_conv: np.ndarray, ring: np.ndarray, ring_pos: int,
                          u_in: np.ndarray) -> tuple[np.ndarray, int]:
    """One token of the depthwise causal short conv followed by SiLU.

    ring [conv_k-1][C] holds the previous conv_k-1 inputs; ring_pos is the
    slot of the oldest.  Reading oldest to newest, tap t (t = 0..conv_k-2)
    meets ring[(ring_pos + t) mod (conv_k-1)] and tap conv_k-1 meets u_in.
    The oldest slot then takes u_in and ring_pos advances by one ("causal
    conv + SiLU with the ring advancing", section "What the PR does").
    ring is updated in place; returns (silu(conv), new ring_pos).
    """
    kk = w_conv.shape[1]
    nslot = kk - 1
    acc = np.zeros(u_in.shape[0], F64)
    for t in range(nslot):
        acc = acc + w_conv[:, t].astype(F64) * ring[(ring_pos + t) % nslot]
    acc = acc + w_conv[:, kk - 1].astype(F64) * u_in
    ring[ring_pos] = u_in
    return silu(acc), (ring_pos + 1) % nslot


def l2_normalize(x: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(sum(x^2) + eps), in double with eps inside the root."""
    x = np.asarray(x, F64)
    return x / np.sqrt(np.sum(x * x) + eps)


def normalize_qk(q: np.ndarray, k: np.ndarray, l2_eps: float, q_scale: float) -> tuple[np.ndarray, np.ndarray]:
    """The per-head L2 norms of q and k (eps inside the root, double), then
    the query scale on the normalised q only: returns (q_scale * q / |q|, k / |k|)."""
    return l2_normalize(q, l2_eps) * F64(q_scale), l2_normalize(k, l2_eps)


def gated_delta_rule_step(S: np.ndarray, q: np.ndarray, k: np.ndarray, v: np.ndarray,
                          g, beta: float) -> tuple[np.ndarray, np.ndarray]:
    """One token of the gated delta rule for one value head, in the page's order.

    1. decay:      S <- exp(g) * S, g a scalar (one gate per head); or, with a
                   per-key-channel gate g[dk] (the gate of the page's KDA
                   engines, "Where this goes next"), row i of S (key index i)
                   is scaled by exp(g[i]): S <- diag(exp(g)) S
    2. delta:      delta = beta * (v - S^T k)   (against the decayed state)
    3. write-back: S <- S + k delta^T
    4. readout:    o = S^T q                     (over the updated state)
    Returns (new S, o).
    """
    g = np.asarray(g, F64)
    S = (np.exp(g) * S) if g.ndim == 0 else (np.exp(g)[:, None] * S)
    kv = S.T @ k
    delta = F64(beta) * (v - kv)
    S = S + np.outer(k, delta)
    o = S.T @ q
    return S, o


def gated_rmsnorm(o: np.ndarray, z: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm of one head's output, times the norm weight, times silu(z)."""
    o = np.asarray(o, F64)
    rms = np.sqrt(np.mean(o * o) + eps)
    return o / rms * w.astype(F64) * silu(np.asarray(z, F64))


class OracleLayer:
    """One gated-DeltaNet layer for a batch of independent sequences, float64.

    The layer object of the page (section "What the PR does") holds the conv
    ring, the recurrent state and the weights; here they live in host
    float64 arrays.  ``step`` advances every sequence by one token.
    """

    def __init__(self, cfg, weights, state):
        self.cfg = cfg
        self.w = weights
        # float64 copies of the int8 matrices (exact), made once per layer
        self.w_in64 = weights.w_in.astype(F64)
        self.w_out64 = weights.w_out.astype(F64)
        self.w_ab64 = weights.w_ab.astype(F64) if getattr(cfg, "device_gates", False) else None
        self.S = np.array(state.S, dtype=F64, copy=True)
        self.ring = np.array(state.ring, dtype=F64, copy=True)
        self.ring_pos = np.array(state.ring_pos, dtype=np.int64, copy=True)

    def step(self, x: np.ndarray, g: np.ndarray | None = None, beta: np.ndarray | None = None,
             trace: dict | None = None) -> np.ndarray:
        """x [B][hidden], g [B][n_v_heads] (or [B][n_v_heads][dk] with the
        per-key gate), beta [B][n_v_heads] -> out [B][hidden] (float64).

        If ``trace`` is a dict it receives the intermediates: "y" (in_proj
        output), "u" (conv+SiLU output), "o" (readout per head) and "normed".

        With device gates (cfg.device_gates) g and beta are not given: the
        layer's a/b gate projections (int8 rows, one scale per row) of x give
        a [B][heads] (or [B][heads][dk]) and b [B][heads], and gate_transform
        turns them into g and beta.
        """
        c, w = self.cfg, self.w
        B = x.shape[0]
        if getattr(c, "device_gates", False):
            if g is not None or beta is not None:
                raise ValueError("a layer with device gates takes no g / beta")
            ab = int8_rowscaled_gemv(self.w_ab64, w.s_ab, x)          # [B][gate_rows]
            na = c.n_v_heads * c.gate_width
            a = ab[:, :na].reshape((B, c.n_v_heads) + ((c.dk,) if c.gate_width > 1 else ()))
            g, beta = gate_transform(a, ab[:, na:], w.gate_A)
        qk, C = c.qk_dim, c.conv_ch
        group = c.n_v_heads // c.n_qk_heads
        y = int8_rowscaled_gemv(self.w_in64, w.s_in, x)     # [B][in_rows]
        normed = np.zeros((B, c.v_dim), F64)
        u_all = np.zeros((B, C), F64)
        o_all = np.zeros((B, c.n_v_heads, c.dv), F64)
        for b in range(B):
            qkv, z = y[b, :C], y[b, C:]
            u, self.ring_pos[b] = causal_conv_silu_step(w.w_conv, self.ring[b], int(self.ring_pos[b]), qkv)
            u_all[b] = u
            q_all = u[0:qk].reshape(c.n_qk_heads, c.dk)
            k_all = u[qk:2 * qk].reshape(c.n_qk_heads, c.dk)
            v_all = u[2 * qk:].reshape(c.n_v_heads, c.dv)
            for h in range(c.n_v_heads):
                hq = h // group
                qh, kh = normalize_qk(q_all[hq], k_all[hq], c.l2_eps, c.qscale)
                self.S[b, h], o = gated_delta_rule_step(self.S[b, h], qh, kh, v_all[h],
                                                        g[b, h], beta[b, h])
                o_all[b, h] = o
                normed[b, h * c.dv:(h + 1) * c.dv] = gated_rmsnorm(
                    o, z[h * c.dv:(h + 1) * c.dv], w.w_norm, c.norm_eps)
        if trace is not None:
            trace.update(y=y, u=u_all, o=o_all, normed=normed)
        return int8_rowscaled_gemv(self.w_out64, w.s_out, normed)


def prefill(layer: "OracleLayer", x: np.ndarray, g: np.ndarray | None = None,
            beta: np.ndarray | None = None) -> np.ndarray:
    """A prompt: x [B][S][hidden] (g [B][S][heads](dk), beta [B][S][heads],
    or None with device gates) through the layer token by token, the
    definition of processing S tokens; returns out [B][S][hidden]."""
    B, S = x.shape[0], x.shape[1]
    out = np.zeros((B, S, x.shape[2]), F64)
    for t in range(S):
        out[:, t] = layer.step(x[:, t], None if g is None else g[:, t], None if beta is None else beta[:, t])
    return out


def rms_prenorm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """Unweighted RMSNorm of each row, used between the layers of a stack."""
    x = np.asarray(x, F64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def stack_step(layers: list[OracleLayer], x: np.ndarray, gates) -> np.ndarray:
    """One token through a stack: x_{l+1} = x_l + layer_l(rms_prenorm(x_l))."""
    h = np.asarray(x, F64)
    for layer, (g, beta) in zip(layers, gates):
        h = h + layer.step(rms_prenorm(h), g, beta)
    return h
