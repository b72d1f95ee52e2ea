"""The torch-tensor wrappers (packed_causal_conv1d_fn, causal_conv1d_update)
reject what the C ABI would misread before any pointer reaches the library:
wrong dtypes (int64 metadata would be read as int32), shapes, a mis-shaped
`out`, and tensors that are not on x's CUDA device. Run on the CPU: the
checks raise before the library is loaded or a kernel launched."""

from __future__ import annotations

import pytest
import torch

import linear_attention_prefill_varlen_gb300 as pkg

DIM, PART, T, N, LINES = 256, 128, 10, 3, 5


def _prefill(**over):
    a = dict(x=torch.zeros(T, DIM, dtype=torch.bfloat16),
             weight=torch.zeros(DIM, 4), bias=torch.zeros(DIM),
             conv_states=torch.zeros(LINES, DIM, 3),
             query_start_loc=torch.tensor([0, 3, 7, T], dtype=torch.int32),
             cache_indices=torch.tensor([0, 2, 4], dtype=torch.int32),
             has_initial_state=torch.ones(N, dtype=torch.bool))
    a.update(over)
    return a


def _call_prefill(**over):
    a = _prefill(**over)
    out = a.pop("out", None)
    return pkg.packed_causal_conv1d_fn(a["x"], a["weight"], a["bias"], a["conv_states"],
                                       a["query_start_loc"], a["cache_indices"],
                                       a["has_initial_state"], PART, out=out)


@pytest.mark.parametrize("over,exc,words", [
    ({"cache_indices": torch.tensor([0, 2, 4], dtype=torch.int64)}, TypeError, "cache_indices"),
    ({"query_start_loc": torch.tensor([0, 3, 7, T], dtype=torch.int64)}, TypeError,
     "query_start_loc"),
    ({"has_initial_state": torch.ones(N, dtype=torch.float32)}, TypeError, "has_initial_state"),
    ({"cache_indices": torch.tensor([0, 2], dtype=torch.int32)}, ValueError, "needed"),
    ({"has_initial_state": torch.ones(N - 1, dtype=torch.bool)}, ValueError, "needed"),
    ({"cache_indices": torch.tensor([[0, 2, 4]], dtype=torch.int32)}, ValueError, "1-D"),
    ({"x": torch.zeros(T, DIM, dtype=torch.int16)}, TypeError, "x must be"),
    ({"x": torch.zeros(DIM, T, dtype=torch.bfloat16).t()}, ValueError, "unit channel stride"),
    ({"weight": torch.zeros(DIM, 3)}, ValueError, "weight"),
    ({"weight": torch.zeros(DIM, 4, dtype=torch.float64)}, ValueError, "weight"),
    ({"bias": torch.zeros(DIM + 1)}, ValueError, "bias"),
    ({"conv_states": torch.zeros(LINES, DIM, 3, dtype=torch.float16)}, ValueError, "conv_states"),
    ({"out": torch.zeros(2, T + 1, PART, dtype=torch.bfloat16)}, ValueError, "out"),
    ({"out": torch.zeros(2, T, PART, dtype=torch.float16)}, ValueError, "out"),
    ({}, ValueError, "CUDA"),  # well-formed, but on the CPU
])
def test_prefill_wrapper_rejects(over, exc, words):
    with pytest.raises(exc, match=words):
        _call_prefill(**over)


def test_prefill_wrapper_rejects_a_bad_part_dim():
    a = _prefill()
    with pytest.raises(ValueError, match="part_dim"):
        pkg.packed_causal_conv1d_fn(a["x"], a["weight"], a["bias"], a["conv_states"],
                                    a["query_start_loc"], a["cache_indices"],
                                    a["has_initial_state"], 96)


@pytest.mark.parametrize("ci,exc,words", [
    (torch.tensor([0, 1, 2, 3], dtype=torch.int64), TypeError, "cache_indices"),
    (torch.tensor([0, 1, 2], dtype=torch.int32), ValueError, "needed"),
    (torch.tensor([0, 1, 2, 3], dtype=torch.int32), ValueError, "CUDA"),
])
def test_update_wrapper_rejects(ci, exc, words):
    x = torch.zeros(4, DIM, dtype=torch.bfloat16)
    with pytest.raises(exc, match=words):
        pkg.causal_conv1d_update(x, torch.zeros(LINES, DIM, 3), torch.zeros(DIM, 4),
                                 torch.zeros(DIM), ci, PART)


@pytest.mark.parametrize("value,code", [
    ("silu", pkg.KDA_ACT_SILU), ("swish", pkg.KDA_ACT_SILU), (True, pkg.KDA_ACT_SILU),
    (None, pkg.KDA_ACT_NONE), (False, pkg.KDA_ACT_NONE), ("none", pkg.KDA_ACT_NONE),
    ("identity", pkg.KDA_ACT_NONE),
])
def test_activation_values_accepted(value, code):
    assert pkg.activation_code(value) == code


@pytest.mark.parametrize("value", ["SiLU", "gelu", "relu", "", 1, 0, 1.0, "Silu "])
def test_activation_values_rejected(value):
    with pytest.raises(ValueError, match="activation"):
        pkg.activation_code(value)
    a = _prefill()
    with pytest.raises(ValueError, match="activation"):  # before any other check
        pkg.packed_causal_conv1d_fn(a["x"], a["weight"], a["bias"], a["conv_states"],
                                    a["query_start_loc"], a["cache_indices"],
                                    a["has_initial_state"], PART, activation=value)
    with pytest.raises(ValueError, match="activation"):
        pkg.causal_conv1d_update(torch.zeros(4, DIM, dtype=torch.bfloat16),
                                 torch.zeros(LINES, DIM, 3), torch.zeros(DIM, 4),
                                 torch.zeros(DIM), torch.zeros(4, dtype=torch.int32), PART,
                                 activation=value)
