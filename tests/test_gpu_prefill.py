"""GPU parity of dn_prefill (a prompt of S tokens per sequence in one call)
against the oracle stepping the same tokens one by one: every token's output,
and the state, the conv ring and its positions after the prompt (and after
decode steps that follow it), within the same 2e-3 bar as the decode step."""
import numpy as np
import pytest

from gated_deltanet_hybrid_gb300.inputs import SHAPE_35B, TINY, WORKLOADS, DNConfig, custom_workload

from harness import REL_TOL, run_prefill_parity

pytestmark = pytest.mark.gpu


def _assert_ok(w):
    assert w["out"] <= REL_TOL, w
    assert w["S"] <= REL_TOL, w
    assert w["ring"] <= REL_TOL, w
    assert w["ring_pos_equal"], w


def test_prefill_49_token_prompt_35b():
    """The 30-layer stack's prompt length (49 tokens) on the 35B-shape layer
    at batch 1: one block of 49 columns (tensor-core projections, the chunked
    recurrence on the CUDA cores over a chunk of 32 tokens and one of 17)."""
    wl = custom_workload("pf49", SHAPE_35B, batch=1, steps=49, seed=3)
    _assert_ok(run_prefill_parity(wl, 49, decode_after=3))


def test_prefill_2048_token_prompt_batch8():
    """The long-prompt workload as one prompt: batch 8, 2048 tokens with
    exp(g) in [0.9, 1] (32 blocks of 8 x 64 columns; the chunked recurrence
    on the tensor cores), sequences 0 and 7 recomputed by the oracle."""
    wl = WORKLOADS["long_prompt_b8"]
    _assert_ok(run_prefill_parity(wl, 2048, sample=np.array([0, 7])))


@pytest.mark.parametrize("batch,n_tokens", [(1, 96), (2, 70)])
def test_prefill_chunked_recurrence_random_state(batch, n_tokens):
    """The chunked recurrence on the CUDA cores (128-dim heads, one decay per
    head, fewer (value head, sequence) pairs than SMs) from a
    random initial state: whole chunks (96 = 3 x 32 tokens in one block) and
    a ragged last chunk (2 x 70 columns: 70 = 2 x 32 + 6 tokens)."""
    cfg = DNConfig(hidden=256, n_qk_heads=2, n_v_heads=4, dk=128, dv=128)
    wl = custom_workload("pfc", cfg, batch=batch, steps=n_tokens, seed=90 + n_tokens, init_std=0.05)
    _assert_ok(run_prefill_parity(wl, n_tokens, decode_after=2))


@pytest.mark.parametrize("shape,batch,n_tokens,gates", [
    ("35b", 5, 70, {}),
    ("small", 40, 13, {}),
    ("small", 40, 13, {"device_gates": True}),
    ("small", 40, 13, {"key_gate": True}),
])
def test_prefill_many_sequences_random_state(shape, batch, n_tokens, gates):
    """Blocks of many sequences on 128-wide heads, from a random initial
    state: the fused partial-sum / conv / norm / ring kernel (one CTA per
    in_proj row tile and sequence) and, with one decay per head, the chunked
    recurrence on the tensor cores.  35B shape at batch 5: one block of 70
    tokens, two whole chunks and a ragged one of 6 (sequences 0 and 4
    recomputed by the oracle).  Four value heads at batch 40: blocks of 12
    and 1 tokens, with the caller's gates, gates
    from the layer's a/b rows, and per-key-channel gates (whose recurrence
    stays token-serial)."""
    if shape == "35b":
        cfg, sample = SHAPE_35B, np.array([0, 4])
    else:
        cfg = DNConfig(hidden=256, n_qk_heads=2, n_v_heads=4, dk=128, dv=128, **gates)
        sample = np.array([0, 17, 39])
    wl = custom_workload("pftc", cfg, batch=batch, steps=n_tokens, seed=700 + batch, init_std=0.05)
    _assert_ok(run_prefill_parity(wl, n_tokens, sample=sample, decode_after=2))


@pytest.mark.parametrize("batch,n_tokens", [(1, 1), (1, 7), (3, 200), (5, 60), (64, 9), (600, 2)])
def test_prefill_tiny_blocks(batch, n_tokens):
    """Block shapes: one token (the CUDA-core projections), a few columns,
    ragged last blocks (3 x 200 -> 170 + 30 tokens), 64 sequences, more than
    512 sequences (two sequence groups); random initial state, so the first
    tokens' convolution reads the ring."""
    wl = custom_workload("pft", TINY, batch=batch, steps=n_tokens, seed=40 + batch, init_std=0.1)
    sample = np.array(sorted({0, batch // 2, batch - 1}))
    _assert_ok(run_prefill_parity(wl, n_tokens, sample=sample, decode_after=2))


@pytest.mark.parametrize("dims", [
    dict(hidden=256, n_qk_heads=1, n_v_heads=2, dk=256, dv=128, conv_k=3),
    dict(hidden=128, n_qk_heads=2, n_v_heads=6, dk=64, dv=32, conv_k=2),
    dict(hidden=256, n_qk_heads=2, n_v_heads=4, dk=32, dv=256, conv_k=5),
    dict(hidden=256, n_qk_heads=2, n_v_heads=4, dk=128, dv=128, key_gate=True),
    dict(hidden=256, n_qk_heads=2, n_v_heads=4, dk=128, dv=128, device_gates=True),
    dict(hidden=256, n_qk_heads=2, n_v_heads=4, dk=32, dv=32, key_gate=True, device_gates=True),
])
def test_prefill_other_dimensions_and_gates(dims):
    cfg = DNConfig(**dims)
    wl = custom_workload("pfd", cfg, batch=3, steps=40, seed=60, init_std=0.05)
    _assert_ok(run_prefill_parity(wl, 40, decode_after=2))


@pytest.mark.parametrize("batch,n_tokens", [(1, 1), (1, 5), (1, 49)])
def test_prefill_int4(batch, n_tokens):
    """A prompt on an int4 layer: one column (the int4 GEMV), 5 and 49
    columns (tensor cores on the int8 expansion; the chunked recurrence with
    a partial chunk, and a full and a partial one)."""
    cfg = DNConfig(hidden=2048, n_qk_heads=16, n_v_heads=32, dk=128, dv=128, int4=True)
    wl = custom_workload("pf_i4", cfg, batch=batch, steps=n_tokens, seed=470 + n_tokens, init_std=0.02)
    _assert_ok(run_prefill_parity(wl, n_tokens, decode_after=2))
