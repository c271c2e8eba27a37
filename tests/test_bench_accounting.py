"""The bench's byte accounting (the roofline numerators) against the per-unit
figures worked out by hand from the tensor shapes, and the stored ncu DRAM
traffic against the current prefill kernel source.  CPU only."""
import bench
from selective_state_space_131_b300 import inputs


def test_prefill_bytes_siso_workload():
    # per token and head (SISO, N = P = 64, bf16): x + y 2 * 128, B + C 2 * 128,
    # theta 32 * 2, dt 4, lambda 4 = 584 B; plus A (32 * 4) and the fp32 final
    # state (8 * 32 * 64 * 64 * 4)
    tokens = 8 * 8192 * 32
    expect = tokens * 584 + 32 * 4 + 8 * 32 * 64 * 64 * 4
    assert expect == 1_228_931_200
    assert bench.scan_bytes(inputs.WORKLOADS[inputs.SISO]) == expect


def test_prefill_bytes_ssd_equivalent_workload():
    # N = 128, no lambda, no theta, bf16: x read and y written (2 * 128 B), B and C
    # read (2 * 256 B), dt 4
    tokens = 8 * 4096 * 32
    per_token = 64 * 2 * 2 + 128 * 2 * 2 + 4
    expect = tokens * per_token + 32 * 4 + 8 * 32 * 128 * 64 * 4
    assert bench.scan_bytes(inputs.WORKLOADS[inputs.SSD_EQUIV]) == expect


def test_decode_bytes_per_step():
    # per (b, h): the fp32 state read and written (2 * 64 * 64 * 4), x / prev_x / y
    # (3 * R * 64 * 4), B / C / prev_B (3 * R * 64 * 4), theta (32 * 4), dt + lambda (8)
    units = 256 * 32
    for R, per_unit in ((1, 34_440), (4, 39_048)):
        assert 2 * 64 * 64 * 4 + 3 * R * 64 * 4 + 3 * R * 64 * 4 + 32 * 4 + 8 == per_unit
        shape = inputs.DecodeShape(**{**inputs.WORKLOADS[inputs.DECODE].__dict__, "rank": R})
        assert bench.decode_bytes(shape) == units * per_unit


def test_backward_bytes_siso_workload():
    # the forward's inputs and their gradients (2 * 584 per token), dy (128), the
    # fp32 dfinal, A and dA
    tokens = 8 * 8192 * 32
    expect = tokens * (2 * 584 + 128) + 8 * 32 * 64 * 64 * 4 + 2 * 32 * 4
    assert bench.bwd_bytes(inputs.WORKLOADS[inputs.SISO]) == expect == 2_722_103_552


def test_stored_prefill_traffic_matches_the_kernel_source():
    """The ncu DRAM bytes stored for the timed workload belong to the current
    source of the prefill kernel (else the bench reports null), and they do not
    exceed the algorithmic bytes: nothing is read twice."""
    traffic = bench.ncu_traffic(inputs.SISO)
    assert traffic is not None
    assert traffic <= bench.scan_bytes(inputs.WORKLOADS[inputs.SISO])
