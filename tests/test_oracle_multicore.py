"""The all-core timing harness runs the unchanged oracle on channel blocks:
its blocks, put together, are exactly the whole-batch call."""

from __future__ import annotations

import numpy as np

import oracle
import pins
from oracle import multicore


def test_channel_blocks_tile_the_channels():
    for dim, parts in [(4608, 16), (384, 7), (64, 64), (5, 16), (3264, 1)]:
        blocks = multicore.channel_blocks(dim, parts)
        assert blocks[0][0] == 0 and blocks[-1][1] == dim
        assert all(a[1] == b[0] for a, b in zip(blocks, blocks[1:]))
        assert all(c1 > c0 for c0, c1 in blocks)
        assert len(blocks) == min(parts, dim)


def test_pool_updates_the_state_as_one_call():
    b = pins.small_batch(901, [5, 1, 40, 2], dim=192, part_dim=64, null_count=1,
                         cache_lines=7, his_p=0.5)
    want = b.conv_states.copy()
    oracle.packed_conv1d(b.x_buf, b.col_offset, b.dim, b.part_dim, b.weight, b.bias, want,
                         b.cache_indices, b.has_initial_state, b.query_start_loc,
                         b.null_block_id, b.activation)
    with multicore.OraclePool(b, procs=3) as pool:
        assert len(pool.workers) == 3
        assert pool.run(1) > 0
        got = pool.states()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_blocks_reassemble_the_whole_output():
    b = pins.small_batch(902, [9, 3, 30], dim=256, part_dim=128, null_count=0, cache_lines=5)
    whole = oracle.packed_conv1d_ex(b.x_buf, oracle.DTYPE_BF16, b.col_offset, b.dim, b.part_dim,
                                    b.weight, b.bias, b.conv_states.copy(), b.cache_indices,
                                    b.has_initial_state, b.query_start_loc, b.null_block_id,
                                    b.activation)["out"]
    flat = np.concatenate(list(whole), axis=1)  # (tokens, dim): planes side by side
    st = b.conv_states.copy()
    for c0, c1 in multicore.channel_blocks(b.dim, 5):
        part = oracle.packed_conv1d_ex(b.x_buf, oracle.DTYPE_BF16, b.col_offset + c0, c1 - c0,
                                       c1 - c0, b.weight[c0:c1], b.bias[c0:c1], st[:, c0:c1, :],
                                       b.cache_indices, b.has_initial_state, b.query_start_loc,
                                       b.null_block_id, b.activation)["out"]
        assert np.array_equal(part[0], flat[:, c0:c1])
