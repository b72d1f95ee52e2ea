"""The algorithmic byte count behind every GB/s figure, against values worked
out by hand from its definition: x read once and the planes written once
(2 bytes each for bf16), 12 bytes per channel for each state line read (when
the sequence has an initial state) and written (fp32 width 3; 6 for bf16),
16 bytes per channel of taps and 4 of bias.  Halo re-reads are not counted."""

from __future__ import annotations

import numpy as np

import workloads


def test_named_workloads():
    # 16K x 4608 prefill, one sequence with its state: 4*T*D + 24*D + 20*D
    assert workloads.algorithmic_bytes(workloads.long16k()) == \
        4 * 16384 * 4608 + 24 * 4608 + 20 * 4608 == 302_192_640
    # 4 x 8192 tokens of 3264 channels, his = [1, 0, 1, 0], no bias
    assert workloads.algorithmic_bytes(workloads.large_nobias()) == \
        4 * 32768 * 3264 + 12 * 3264 * 2 + 12 * 3264 * 4 + 16 * 3264 == 428_106_240
    # 64 tokens of 384 channels
    assert workloads.algorithmic_bytes(workloads.tiny()) == \
        4 * 64 * 384 + 24 * 384 + 20 * 384 == 115_200
    # decode: 1024 one-token sequences, every line read and written
    assert workloads.algorithmic_bytes(workloads.decode()) == \
        4 * 1024 * 4608 + 24 * 4608 * 1024 + 20 * 4608 == 132_212_736
    # the same with the state stored as bf16: half the state bytes
    assert workloads.algorithmic_bytes(workloads.decode_bf16_state()) == \
        4 * 1024 * 4608 + 12 * 4608 * 1024 + 20 * 4608 == 75_589_632


def test_empty_null_and_fresh_sequences():
    """Lengths [3, 0, 2, 4] on 64 channels: the empty sequence moves nothing,
    the null-block one only its rows, the one without history writes its
    line but reads none."""
    b = workloads.make_batch("bytes", 1, [3, 0, 2, 4], 64, 64, 64, 6)
    b.cache_indices = np.array([0, 1, -1, 2], dtype=np.int32)
    b.null_block_id = -1
    b.has_initial_state = np.array([1, 1, 1, 0], dtype=np.uint8)
    rows = 3 + 2 + 4
    want = (2 * 2 * rows * 64      # x in, planes out
            + 12 * 64 * 1          # reads: sequence 0 only
            + 12 * 64 * 2          # writes: sequences 0 and 3
            + 16 * 64 + 4 * 64)    # taps, bias
    assert workloads.algorithmic_bytes(b) == want
    b.bias = None
    assert workloads.algorithmic_bytes(b) == want - 4 * 64


def test_fp32_x_counts_four_bytes_per_element():
    b = workloads.make_batch("bytes32", 2, [5], 64, 64, 64, 2, x_dtype="f32")
    b.has_initial_state[:] = 1
    assert workloads.algorithmic_bytes(b) == 2 * 4 * 5 * 64 + 24 * 64 + 20 * 64
