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


class _Torch152:
    """Stands in for torch.cuda's device query: a GB300 has 152 SMs."""

    class cuda:
        @staticmethod
        def current_device():
            return 0

        @staticmethod
        def get_device_properties(_):
            return type("Props", (), {"multi_processor_count": 152})()


def test_prefill_blocks_and_kernel_counts():
    """The prompt bench's launch claim: dn_prefill cuts a prompt into blocks
    of up to 512 token columns (512 // B tokens for B sequences), and a block
    launches gather, (pack +) in_proj, steps 2-4, the recurrence, the gated
    norm, the out_proj and its reduction, where steps 2-4 are one kernel for
    128-wide heads once (in_proj row tiles x sequences) covers the SMs."""
    blocks = list(bench.prefill_blocks(8, 2048))
    assert len(blocks) == 32 and set(blocks) == {(8, 512)}
    assert list(bench.prefill_blocks(1, 49)) == [(1, 49)]
    assert list(bench.prefill_blocks(3, 200)) == [(3, 510), (3, 90)]  # 170 + 30 tokens
    assert list(bench.prefill_blocks(600, 2)) == [(512, 512), (512, 512), (88, 176)]  # 1 token per block
    t = _Torch152
    # 35B shape: 96 row tiles, so one sequence (96 CTAs) keeps the three kernels
    assert bench.prefill_block_kernels(SHAPE_35B, 8, 512, t) == 1 + 2 + 1 + 4
    assert bench.prefill_block_kernels(SHAPE_35B, 2, 512, t) == 1 + 2 + 1 + 4
    assert bench.prefill_block_kernels(SHAPE_35B, 1, 49, t) == 1 + 2 + 3 + 4
    assert bench.prefill_block_kernels(SHAPE_35B, 1, 1, t) == 1 + 1 + 3 + 4  # the GEMV, no pack
    # 32-wide heads never fuse steps 2-4
    assert bench.prefill_block_kernels(TINY, 256, 256, t) == 1 + 2 + 3 + 4
