"""Shared helpers for the GPU parity tests: upload a host batch, run the
library through its C ABI, run the oracle on the same bytes, compare."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import pins
import workloads

SENTINEL = -1  # int16 view of the bf16 pattern 0xFFFF (a NaN no conv produces)


def state_to_device(states: np.ndarray, dev) -> torch.Tensor:
    """Host conv states (float32, or uint16 bf16 bits) as a device tensor of
    the same bytes (float32 or bfloat16), strides kept."""
    if states.dtype == np.uint16:
        return torch.from_numpy(states.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(states).to(dev)


def state_dtype_of(states: torch.Tensor) -> int:
    """The kda_dtype_t of a device conv-state tensor."""
    return 0 if states.dtype == torch.bfloat16 else 2  # KDA_DTYPE_BF16 / KDA_DTYPE_F32


def state_to_host(states: torch.Tensor) -> np.ndarray:
    """The inverse of state_to_device, as a contiguous array."""
    if states.dtype == torch.bfloat16:
        return states.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    return states.contiguous().cpu().numpy()


def ordered_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers that step by one per representable value
    (sign-magnitude to two's-complement order; +0 and -0 are one apart)."""
    b = bits.astype(np.int32)
    return np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + (b & 0x7FFF))


def is_nan_bf16(bits: np.ndarray) -> np.ndarray:
    return ((bits & 0x7F80) == 0x7F80) & ((bits & 0x007F) != 0)


def ulp_diff(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """|ordered(got) - ordered(want)|, with NaN == NaN counted as 0."""
    d = np.abs(ordered_bf16(got) - ordered_bf16(want))
    both_nan = is_nan_bf16(got) & is_nan_bf16(want)
    return np.where(both_nan, 0, d)


class DeviceBatch:
    """A workloads.Batch copied to the GPU (the same bytes as the host copy)."""

    def __init__(self, b: workloads.Batch, device="cuda", preact: bool = False):
        self.b = b
        dev = torch.device(device)
        self.x_buf = torch.from_numpy(b.x_buf.view(np.int16)).to(dev)
        self.weight = torch.from_numpy(b.weight).to(dev)
        self.bias = None if b.bias is None else torch.from_numpy(b.bias).to(dev)
        self.conv_states = state_to_device(b.conv_states, dev)
        self.cache_indices = torch.from_numpy(b.cache_indices).to(dev)
        self.has_initial_state = torch.from_numpy(b.has_initial_state).to(dev)
        self.query_start_loc = torch.from_numpy(b.query_start_loc).to(dev)
        shape = (b.dim // b.part_dim, b.tokens, b.part_dim)
        if preact:
            self.out = torch.full(shape, float("nan"), dtype=torch.float32, device=dev)
        else:
            self.out = torch.full(shape, SENTINEL, dtype=torch.int16, device=dev)

    @property
    def x_ptr(self) -> int:
        return self.x_buf.data_ptr() + 2 * self.b.col_offset

    def args(self):
        b = self
        return (self.x_ptr, self.b.row_stride, self.b.tokens, self.b.dim, self.b.part_dim,
                b.weight, b.bias, b.conv_states, b.cache_indices, b.has_initial_state,
                b.query_start_loc, self.b.num_seqs, self.b.null_block_id)

    def run(self, stream=None) -> None:
        """kda_packed_conv1d; kda_packed_conv1d_ex with a bf16-state layout
        when the batch's state is bf16."""
        import linear_attention_prefill_varlen_gb300 as pkg

        if self.conv_states.dtype == torch.bfloat16:
            st = self.conv_states
            lay = pkg.make_layout(pkg.KDA_DTYPE_BF16, st.size(2), st.stride(), (4, 1),
                                  pkg.KDA_DTYPE_BF16)
            pkg.kda_packed_conv1d_ex(*self.args(), self.b.activation, self.out, lay, stream)
        else:
            pkg.kda_packed_conv1d(*self.args(), self.b.activation, self.out, stream)

    def run_preact(self, stream=None) -> None:
        import linear_attention_prefill_varlen_gb300 as pkg

        pkg.kda_packed_conv1d_preact_f32(*self.args(), self.out, stream)

    def out_bits(self) -> np.ndarray:
        return self.out.cpu().numpy().view(np.uint16)

    def states(self) -> np.ndarray:
        return state_to_host(self.conv_states)


def oracle_run(b: workloads.Batch, want_preact: bool = False) -> tuple[dict, np.ndarray]:
    """Runs the oracle on a copy of b's state; returns (result, updated states)."""
    st = b.conv_states.copy()
    if st.dtype == np.uint16:  # bf16 state: the general-layout oracle
        return pins.run_oracle_ex(b, states=st, want_preact=want_preact), st
    res = oracle.packed_conv1d(b.x_buf, b.col_offset, b.dim, b.part_dim, b.weight, b.bias, st,
                               b.cache_indices, b.has_initial_state, b.query_start_loc,
                               b.null_block_id, b.activation, want_preact=want_preact)
    return res, st


def assert_states_equal(got: np.ndarray, want: np.ndarray) -> None:
    assert got.dtype == want.dtype and got.shape == want.shape
    g, w = (got.view(np.uint32), want.view(np.uint32)) if got.dtype == np.float32 else (got, want)
    if not np.array_equal(g, w):
        bad = np.argwhere(g != w)
        raise AssertionError(f"{len(bad)} conv-state words differ; first at {bad[0].tolist()}")


def assert_outputs_match(got: np.ndarray, want: np.ndarray, activation: int) -> dict:
    """activation 0: bit-exact.  SiLU: within 1 bf16 ulp.  Rows the oracle left
    at the sentinel must still hold it.  Returns mismatch statistics."""
    d = ulp_diff(got, want)
    stats = {"mismatches": int(np.count_nonzero(d)), "max_ulp": int(d.max()) if d.size else 0}
    if d.size and stats["mismatches"]:
        stats["first"] = np.argwhere(d != 0)[0].tolist()
    untouched = want == 0xFFFF
    assert np.array_equal(got[untouched], want[untouched]), "rows outside sequences written"
    limit = 0 if activation == 0 else 1
    assert stats["max_ulp"] <= limit, stats
    return stats
