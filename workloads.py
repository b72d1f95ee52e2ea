"""Seeded synthetic inputs for the packed varlen causal conv1d.

This module only draws random numbers and lays them out; it holds none of
the conv's arithmetic.  The same host arrays feed the CPU oracle and (copied
to the device) the CUDA library, so both sides see identical bytes.

Every draw comes from a CPU ``torch.Generator`` seeded per workload, in the
order written in ``make_batch``.  bf16 inputs are fp32 normal samples
converted by torch's own ``.to(torch.bfloat16)``.

Workloads (shapes from the Kimi-K3 KDA in_proj as the vLLM page
"vllm.models.kimi_k3.nvidia.ops.kda_conv" sizes it: 3 x 1536 channels, 16K
token prefill chunks, row-strided bf16 slices of a wider projection):

  tiny          1 x 64 tokens, dim 384 = 3 x 128, dense rows, SiLU, seed 0
  varlen        8 sequences, lengths U[1,512], dim 4608 = 3 x 1536, row stride
                6400, one padding sequence (null block), his ~ Bernoulli(0.5),
                SiLU, seed 1
  long16k       1 x 16384 tokens, dim 4608, row stride 6400, SiLU, seed 2
  short_decode  256 sequences with lengths U[1,128] followed by 1024 one-token
                (decode-shaped) sequences in one call, dim 4608, row stride
                6400, 2048 cache lines, his ~ Bernoulli(0.8), SiLU, seed 3
  large_nobias  4 x 8192 tokens, dim 3264 = 3 x 1088, dense rows, x ~ N(0, 2^2),
                weight U(-1, 1), no bias, no activation, seed 4
  decode        1024 sequences of 1 token (a decode step), dim 4608, row stride
                6400, 2048 cache lines, every sequence with an initial state, seed 5
  decode_bf16_state  the decode draws with the conv state rounded to bf16
  spec_decode   1024 sequences of 4 tokens (a speculative-decoding verification
                step: one accepted token plus three drafts), dim 4608, row stride
                6400, 2048 cache lines, every sequence with an initial state, seed 6
"""

from __future__ import annotations

from dataclasses import dataclass, field

import re

import numpy as np
import torch

NULL_BLOCK_ID = -1  # the pages do not print the constant; -1 is no valid cache line


@dataclass
class Batch:
    """One call's inputs, as host numpy arrays."""

    name: str
    x_buf: np.ndarray  # (tokens, row_stride) uint16: bf16 bits of the whole in_proj rows
    col_offset: int  # x = x_buf[:, col_offset:col_offset + dim]
    dim: int
    part_dim: int
    weight: np.ndarray  # (dim, 4) float32
    bias: np.ndarray | None  # (dim,) float32
    conv_states: np.ndarray  # (cache_lines, dim, K) float32, or uint16 bf16 bits
    cache_indices: np.ndarray  # (num_seqs,) int32
    has_initial_state: np.ndarray  # (num_seqs,) uint8 (0/1)
    query_start_loc: np.ndarray  # (num_seqs + 1,) int32
    null_block_id: int
    activation: int  # 0 none, 1 SiLU
    seed: int
    notes: dict = field(default_factory=dict)
    x_dtype: str = "bf16"  # storage of x and out: "bf16" / "f16" (uint16 bits) or "f32"

    @property
    def tokens(self) -> int:
        return int(self.x_buf.shape[0])

    @property
    def row_stride(self) -> int:
        return int(self.x_buf.shape[1])

    @property
    def num_seqs(self) -> int:
        return int(self.query_start_loc.size - 1)

    @property
    def cache_lines(self) -> int:
        return int(self.conv_states.shape[0])

    def copy(self) -> "Batch":
        """Deep copy (conv_states is updated in place by a call)."""
        return Batch(
            self.name, self.x_buf.copy(), self.col_offset, self.dim, self.part_dim,
            self.weight.copy(), None if self.bias is None else self.bias.copy(),
            self.conv_states.copy(), self.cache_indices.copy(), self.has_initial_state.copy(),
            self.query_start_loc.copy(), self.null_block_id, self.activation, self.seed,
            dict(self.notes), self.x_dtype)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def _x_storage(t: torch.Tensor, x_dtype: str) -> np.ndarray:
    """fp32 samples stored as the call's x type, by torch's own conversion."""
    if x_dtype == "bf16":
        return bf16_bits(t)
    if x_dtype == "f16":
        return t.to(torch.float16).contiguous().view(torch.int16).numpy().view(np.uint16)
    assert x_dtype == "f32"
    return t.contiguous().numpy().astype(np.float32)


def make_batch(name: str, seed: int, lengths, dim: int, part_dim: int, row_stride: int,
               cache_lines: int, *, col_offset: int = 0, x_std: float = 1.0,
               w_range: float = 0.5, bias_std: float | None = 0.1, activation: int = 1,
               his_p: float = 1.0, his: list[int] | None = None, null_count: int = 0,
               tokens: int | None = None, first_token: int = 0, x_dtype: str = "bf16",
               state_width: int = 3, state_dtype: str = "f32") -> Batch:
    """Draws one batch.

    Draw order: lengths are given; x (tokens, row_stride) ~ N(0, x_std^2);
    weight (dim, 4) ~ U(-w_range, w_range); bias (dim) ~ N(0, bias_std^2) if
    bias_std is not None; conv_states (cache_lines, dim, state_width) ~ N(0, 1),
    kept as float32 or (state_dtype "bf16") rounded to bf16 bits by torch;
    cache_indices = the first num_seqs of a random permutation of the cache
    lines; has_initial_state ~ Bernoulli(his_p) unless given; then
    `null_count` distinct random sequences get NULL_BLOCK_ID as cache index.

    Sequences are packed back to back from `first_token`; `tokens` (default:
    the end of the last sequence) may leave rows after the last sequence that
    no sequence owns.
    """
    g = torch.Generator().manual_seed(seed)
    lengths = [int(v) for v in lengths]
    n = len(lengths)
    qsl = np.zeros(n + 1, dtype=np.int32)
    qsl[0] = first_token
    qsl[1:] = first_token + np.cumsum(np.asarray(lengths, dtype=np.int64))
    total = int(qsl[-1]) if tokens is None else int(tokens)
    assert total >= int(qsl[-1])
    x = _x_storage(torch.randn(total, row_stride, generator=g) * x_std, x_dtype)
    w = ((torch.rand(dim, 4, generator=g) * 2.0 - 1.0) * w_range).numpy().astype(np.float32)
    b = None
    if bias_std is not None:
        b = (torch.randn(dim, generator=g) * bias_std).numpy().astype(np.float32)
    s_draw = torch.randn(cache_lines, dim, state_width, generator=g)
    if state_dtype == "bf16":
        s = bf16_bits(s_draw)
    else:
        assert state_dtype == "f32"
        s = s_draw.numpy().astype(np.float32)
    assert n <= cache_lines
    ci = torch.randperm(cache_lines, generator=g)[:n].numpy().astype(np.int32)
    if his is None:
        hv = (torch.rand(n, generator=g) < his_p).numpy().astype(np.uint8)
    else:
        hv = np.asarray(his, dtype=np.uint8)
    if null_count:
        pos = torch.randperm(n, generator=g)[:null_count].numpy()
        ci[pos] = NULL_BLOCK_ID
    return Batch(name, np.ascontiguousarray(x), col_offset, dim, part_dim, np.ascontiguousarray(w),
                 b, np.ascontiguousarray(s), ci, hv, qsl, NULL_BLOCK_ID, activation, seed,
                 x_dtype=x_dtype)


def _lengths(seed: int, n: int, lo: int, hi: int) -> list[int]:
    g = torch.Generator().manual_seed(seed + 1000)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def tiny(**kw) -> Batch:
    # cache_indices = [2] as the workload fixes it, regardless of the permutation draw.
    b = make_batch("tiny", 0, [64], 384, 128, 384, 4, his=[1], **kw)
    b.cache_indices[:] = 2
    return b


# Each workload takes make_batch's x_dtype / state_width / state_dtype keywords
# for the same draws stored another way (the general-layout measurements).

def varlen(**kw) -> Batch:
    return make_batch("varlen", 1, _lengths(1, 8, 1, 512), 4608, 1536, 6400, 64,
                      his_p=0.5, null_count=1, **kw)


def long16k(**kw) -> Batch:
    return make_batch("long16k", 2, [16384], 4608, 1536, 6400, 8, his=[1], **kw)


def short_decode(**kw) -> Batch:
    lens = _lengths(3, 256, 1, 128) + [1] * 1024
    return make_batch("short_decode", 3, lens, 4608, 1536, 6400, 2048, his_p=0.8, **kw)


def large_nobias(**kw) -> Batch:
    return make_batch("large_nobias", 4, [8192] * 4, 3264, 1088, 3264, 16, x_std=2.0,
                      w_range=1.0, bias_std=None, activation=0, his=[1, 0, 1, 0], **kw)


def decode(**kw) -> Batch:
    """1024 sequences of one token each (a decode step), 2048 cache lines."""
    return make_batch("decode", 5, [1] * 1024, 4608, 1536, 6400, 2048, his_p=1.0, **kw)


def decode_bf16_state(**kw) -> Batch:
    """The decode step with the conv state stored as bf16."""
    return make_batch("decode_bf16_state", 5, [1] * 1024, 4608, 1536, 6400, 2048, his_p=1.0,
                      state_dtype="bf16", **kw)


def spec_decode(**kw) -> Batch:
    """1024 sequences of 4 tokens each, 2048 cache lines."""
    return make_batch("spec_decode", 6, [4] * 1024, 4608, 1536, 6400, 2048, his_p=1.0, **kw)


def skewed(**kw) -> Batch:
    """One 8192-token prompt among 99 sequences of 80 tokens (16,112 tokens,
    128 cache lines): many sequences, one of them long."""
    lens = [80] * 50 + [8192] + [80] * 49
    return make_batch("skewed", 7, lens, 4608, 1536, 6400, 128, his_p=0.8, **kw)


WORKLOADS = {
    "tiny": tiny,
    "varlen": varlen,
    "long16k": long16k,
    "short_decode": short_decode,
    "large_nobias": large_nobias,
    "decode": decode,
    "decode_bf16_state": decode_bf16_state,
    "spec_decode": spec_decode,
    "skewed": skewed,
}


def prefill(tokens: int, **kw) -> Batch:
    """One prefill sequence of `tokens` tokens, otherwise the 16K chunk's shape
    (3 x 1536 channels, row stride 6400, an initial state, 8 cache lines)."""
    return make_batch(f"prefill{tokens}", 2, [tokens], 4608, 1536, 6400, 8, his=[1], **kw)


def decode_batch(n: int, **kw) -> Batch:
    """n sequences of one token each (a decode step), 2n cache lines."""
    return make_batch(f"decode{n}", 5, [1] * n, 4608, 1536, 6400, 2 * n, his_p=1.0, **kw)


_SIZED = re.compile(r"(prefill|decode)([1-9][0-9]{0,6})")


def valid_name(name: str) -> bool:
    return name in WORKLOADS or _SIZED.fullmatch(name) is not None


def by_name(name: str, **kw) -> Batch:
    """A workload of WORKLOADS, or prefill<T> / decode<N> at any size (for
    size sweeps; the same draws as long16k / decode at their own sizes)."""
    if name in WORKLOADS:
        return WORKLOADS[name](**kw)
    m = _SIZED.fullmatch(name)
    if m is None:
        raise KeyError(name)
    n = int(m.group(2))
    return prefill(n, **kw) if m.group(1) == "prefill" else decode_batch(n, **kw)


def algorithmic_bytes(b: Batch) -> int:
    """Bytes a call must move at minimum: x read once, out written once, each
    referenced state line read (if it has an initial state) and written, the
    weight and bias read once.  Halo re-reads are not counted."""
    qsl = b.query_start_loc.astype(np.int64)
    lens = qsl[1:] - qsl[:-1]
    live = lens > 0
    not_null = b.cache_indices != b.null_block_id
    rows = int(lens[live].sum())
    reads = int(np.count_nonzero(live & not_null & (b.has_initial_state != 0)))
    writes = int(np.count_nonzero(live & not_null))
    d = b.dim
    xb = 4 if b.x_dtype == "f32" else 2
    sb = b.conv_states.itemsize * b.conv_states.shape[2]
    return (2 * xb * rows * d + sb * d * reads + sb * d * writes + 16 * d
            + (4 * d if b.bias is not None else 0))
