"""The benchmark's byte model, on the CPU: the algorithmic bytes that the
roofline figures divide by.  The per-step figures of the 35B-shape layer are
fixed by the layer's sizes alone (weights once per step; per sequence the
state read and written, the conv ring's history read and one slot written,
x, out and the two gates), so they are pinned here to the products written
out by hand, and the per-stage model is checked to account for every tensor
of the step."""
from gated_deltanet_hybrid_gb300.inputs import SHAPE_35B, TINY

import bench


def test_35b_step_bytes_by_hand():
    # shared: W_in int8 12288 x 2048, s_in, W_out int8 2048 x 4096, s_out, w_conv 8192 x 4, w_norm 128
    shared = 12288 * 2048 + 12288 * 4 + 2048 * 4096 + 2048 * 4 + 8192 * 4 * 4 + 128 * 4
    assert shared == 33_743_360
    # per sequence: 2 x S (32 x 128 x 128 fp32), ring 3 slots read + 1 written (8192 fp32 each),
    # x and out (2048 fp32 each), g and beta (32 fp32 each)
    per_seq = 2 * 32 * 128 * 128 * 4 + 3 * 8192 * 4 + 8192 * 4 + 2 * 2048 * 4 + 2 * 32 * 4
    assert per_seq == 4_342_016
    assert bench.step_bytes(SHAPE_35B, 1) == shared + per_seq == 38_085_376
    assert bench.step_bytes(SHAPE_35B, 64) == shared + 64 * per_seq == 311_632_384


def test_stage_model_covers_the_step():
    """Every byte of the step model appears in exactly one stage, and the two
    intermediates (the in_proj output, the gated-norm output) once on each
    side of their stage boundary."""
    for cfg in (SHAPE_35B, TINY):
        for B in (1, 8, 64):
            kb = bench.kernel_bytes(cfg, B)
            intermediates = 2 * B * (cfg.in_rows + cfg.v_dim) * 4
            assert sum(kb.values()) == bench.step_bytes(cfg, B) + intermediates
            assert kb["dn_state"] > kb["in_proj"] + kb["out_proj"] or B < 8


def test_state_stage_dominates_at_batch_64():
    """At batch 64 the state stage moves 90 % of the step's bytes: the state
    kernel is the dominant kernel whose roofline the benchmark reports."""
    kb = bench.kernel_bytes(SHAPE_35B, 64)
    assert kb["dn_state"] == 281_166_336
    assert kb["dn_state"] / bench.step_bytes(SHAPE_35B, 64) > 0.9
