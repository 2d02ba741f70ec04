"""The roofline arithmetic of bench.py against figures worked out independently from the layer's shapes:
13,369,344 bytes per MXFP4 expert (gate, up and down: 3 d f / 2 codes + 3 d f / 32 scale bytes), 3.449 GB
for a verify512 layer with every expert touched (weights, fp32 router weight and bias, bf16 x in and out),
and 2.886e12 FLOP for the prefill8192 expert GEMMs (57,344 rows: 49,152 routed + 8,192 shared)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_expert_bytes_match_the_mxfp4_layout():
    wl = synth.WORKLOADS["verify512"]
    assert bench.expert_bytes(wl) == 13_369_344
    # 12,582,912 bytes of E2M1 codes and 786,432 E8M0 bytes
    assert 3 * 4096 * 2048 // 2 == 12_582_912 and 3 * 4096 * 2048 // 32 == 786_432


def test_layer_bytes_of_the_verify_and_hash_layers():
    v = synth.WORKLOADS["verify512"]
    # 257 experts, router weight 256 x 4096 fp32 + 256 biases, x and out 512 x 4096 bf16
    assert bench.layer_bytes(v, 257) == 257 * 13_369_344 + 4_194_304 + 1_024 + 4_194_304 + 4_194_304
    assert bench.layer_bytes(v, 257) == 3_448_505_344
    h = synth.WORKLOADS["hash512"]
    # no router weight; 512 token ids and 512 x 6 table entries instead
    assert bench.layer_bytes(h, 257) == 257 * 13_369_344 + 2 * 4_194_304 + 512 * 4 + 512 * 6 * 4


def test_prefill_gemm_flops():
    p = synth.WORKLOADS["prefill8192"]
    rows = 8192 * 6 + 8192
    fl = bench.gemm_flops(p, rows)
    assert fl["gemm_gate_up"] == 2 * 57_344 * 2 * 2048 * 4096
    assert fl["gemm_gate_up"] + fl["gemm_down"] == 2_886_218_022_912


def test_stage_bytes_count_each_stream_once():
    v = synth.WORKLOADS["verify512"]
    rows = 512 * 7
    sb = bench.stage_bytes(v, 257, rows)
    # gate-up: the weights, the MXFP8 activation rows in, the MXFP8 h rows out
    assert sb["gemm_gate_up"] == 257 * (2 * 2048 * 4096 // 2 + 2 * 2048 * 4096 // 32) + rows * (4096 + 128) + rows * (
        2048 + 64)
    # down: the weights, h in, the weighted rows out as fp16 plus one scale byte per 32 columns
    assert sb["gemm_down"] == 257 * (4096 * 2048 // 2 + 4096 * 2048 // 32) + rows * (2048 + 64) + rows * (8192 + 128)
    # combine: those rows in, the bf16 output
    assert sb["combine"] == rows * (8192 + 128) + 512 * 4096 * 2
    # the MXFP4-activation variant halves the activation and h bytes
    sb4 = bench.stage_bytes(v, 257, rows, "mxfp4")
    assert sb["gemm_gate_up"] - sb4["gemm_gate_up"] == rows * 2048 + rows * 1024
