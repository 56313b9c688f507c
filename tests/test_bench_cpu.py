"""The bench's roofline accounting on the CPU: bytes per expert, FLOP per token and
the bytes of a batch-1 step, against the figures the layer's shape fixes (256
experts, top-8 + 1 shared, H = 2048, F = 512, 64-wide groups with a bf16 scale
and bias each) and against the sizes of the weight arrays the input generator
actually builds."""
import workloads

import bench

FULL = workloads.WORKLOADS["prefill4k"].shape


def test_expert_bytes_full_shape():
    # gate/up: 2F x H nibbles = 1,048,576 B + 2 x (2F x H / 64) bf16 = 131,072 B; down: half of each
    w13, w2 = bench.expert_bytes(FULL)
    assert (w13, w2) == (1_179_648, 589_824)
    assert w13 + w2 == 1_769_472


def test_expert_bytes_equal_generated_arrays():
    d = workloads.make_workload(workloads.WORKLOADS["tiny"])
    n = d["w13_packed"].shape[0]  # E + 1 experts (the shared one last)
    w13 = (d["w13_packed"].nbytes + d["w13_scale"].nbytes + d["w13_bias"].nbytes) // n
    w2 = (d["w2_packed"].nbytes + d["w2_scale"].nbytes + d["w2_bias"].nbytes) // n
    assert bench.expert_bytes(d["workload"].shape) == (w13, w2)


def test_flop_per_token():
    # 2 FLOP per MAC over (k + 1) experts x (gate, up, down) x H x F
    for T in (1, 512, 4096):
        a = bench.algorithmic(FULL, T, 256)
        assert a["step_flops"] / T == 56_623_104


def test_batch1_step_bytes():
    # 8 routed + 1 shared expert's weights, plus x (bf16), the logits (fp32) and out (bf16) of one token
    a = bench.algorithmic(FULL, 1, 8)
    assert a["step_bytes"] == 9 * 1_769_472 + 2048 * 2 + 256 * 4 + 2048 * 2
    assert abs(a["step_bytes"] / 1e6 - 15.93) < 0.01
