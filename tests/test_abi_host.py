"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and its host-only logic (argument checks, launch shape, metadata
validation, empty calls) behaves as documented.  No kernel is launched."""

from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda_conv.h")


@pytest.fixture(scope="module")
def kda():
    from linear_attention_prefill_varlen_gb300 import _binding, _build

    _build.build()
    _binding.lib()
    return _binding


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_conv_entry_point():
    names = declared_functions()
    assert "kda_packed_conv1d" in names
    assert len(names) >= 8, names


def test_library_exports_every_declared_symbol(kda):
    handle = ctypes.CDLL(kda.lib_path())
    missing = [n for n in declared_functions() if not hasattr(handle, n)]
    assert not missing, missing


A16 = 1 << 20  # a fake 16-byte aligned address: never dereferenced by the host checks


def good_args(**over):
    args = dict(x=A16, x_row_stride=6400, tokens=100, dim=4608, part_dim=1536, weight=A16,
                bias=A16, conv_states=A16, cache_indices=A16, has_initial_state=A16,
                query_start_loc=A16, num_seqs=3, activation=1, out=A16)
    args.update(over)
    return args


def check(kda, **over) -> int:
    a = good_args(**over)
    return kda.check_args(a["x"], a["x_row_stride"], a["tokens"], a["dim"], a["part_dim"],
                          a["weight"], a["bias"], a["conv_states"], a["cache_indices"],
                          a["has_initial_state"], a["query_start_loc"], a["num_seqs"],
                          a["activation"], a["out"])


@pytest.mark.parametrize("over,status", [
    ({}, 0),
    ({"bias": None}, 0),
    ({"activation": 0}, 0),
    ({"activation": 2}, 1),
    ({"tokens": -1}, 1),
    ({"num_seqs": -1}, 1),
    ({"x_row_stride": 4600}, 1),
    ({"part_dim": 0}, 1),
    ({"part_dim": 1000}, 2),
    ({"part_dim": 1024}, 2),  # multiple of 64 that does not divide dim
    ({"x": None}, 1),
    ({"weight": None}, 1),
    ({"conv_states": None}, 1),
    ({"cache_indices": None}, 1),
    ({"has_initial_state": None}, 1),
    ({"query_start_loc": None}, 1),
    ({"out": None}, 1),
    ({"x": A16 + 2}, 3),
    ({"x_row_stride": 6404}, 3),
    ({"weight": A16 + 4}, 3),
    ({"bias": A16 + 8}, 3),
    ({"conv_states": A16 + 4}, 3),
    ({"out": A16 + 2}, 3),
    ({"tokens": 0, "x": None, "out": None}, 0),  # empty: nothing is touched
    ({"num_seqs": 0, "query_start_loc": None}, 0),
])
def test_argument_checks(kda, over, status):
    assert check(kda, **over) == status


def test_entry_point_rejects_before_any_cuda_call(kda):
    """Rejected and empty calls return without touching CUDA (safe without a GPU)."""
    with pytest.raises(kda.KdaError) as e:
        kda.kda_packed_conv1d(A16, 6400, 100, 4608, 1000, A16, A16, A16, A16, A16, A16, 3, -1, 1,
                              A16, stream=0)
    assert e.value.status == kda.KDA_ERR_UNSUPPORTED
    with pytest.raises(kda.KdaError) as e:
        kda.kda_packed_conv1d(A16 + 2, 6400, 100, 4608, 1536, A16, A16, A16, A16, A16, A16, 3, -1,
                              1, A16, stream=0)
    assert e.value.status == kda.KDA_ERR_MISALIGNED
    kda.kda_packed_conv1d(A16, 6400, 0, 4608, 1536, A16, A16, A16, A16, A16, A16, 3, -1, 1, A16,
                          stream=0)
    kda.kda_packed_conv1d(A16, 6400, 5, 4608, 1536, A16, A16, A16, A16, A16, A16, 0, -1, 1, A16,
                          stream=0)


def test_status_strings(kda):
    h = kda.lib()
    for s in range(6):
        assert h.kda_status_string(s)
    assert h.kda_status_string(99) == b"unknown status"


@pytest.mark.parametrize("tokens,num_seqs", [(16384, 1), (2430, 8), (18003, 1280), (64, 1),
                                             (1, 1), (100, 400)])
def test_launch_shape_bound(kda, tokens, num_seqs):
    """Programs = ceil(tokens / chunk) + num_seqs: every sequence adds at most
    one partial chunk (the bound of the page's launch)."""
    sh = kda.launch_shape(tokens, 4608, 1536, num_seqs)
    assert sh["chunk"] >= 4
    assert sh["programs"] == -(-tokens // sh["chunk"]) + num_seqs
    # enough threads for every program's channel vectors (at most 8 channels each)
    assert sh["ctas"] * sh["threads"] * 8 >= sh["programs"] * 4608


def test_program_map_covers_every_chunk_once(kda):
    """The map f(s) = floor(qsl[s] / chunk) + s gives each sequence at least
    ceil(len / chunk) programs inside the grid (host model of the device map)."""
    rng = np.random.default_rng(5)
    for trial in range(200):
        n = int(rng.integers(1, 60))
        lens = rng.integers(0, 300, size=n)
        qsl = np.concatenate([[int(rng.integers(0, 50))], lens]).cumsum()
        tokens = int(qsl[-1] + rng.integers(0, 20))
        sh = kda.launch_shape(tokens, 256, 128, n)
        chunk = sh["chunk"]
        f = qsl[:-1] // chunk + np.arange(n)
        f_next = np.append(f[1:], sh["programs"])
        assert (np.diff(f) >= 1).all()
        assert (f_next - f >= -(-lens // chunk)).all()
        assert f[-1] + -(-lens[-1] // chunk) <= sh["programs"]


def test_validate_metadata(kda):
    ok = kda.validate_metadata(torch.tensor([0, 2, 5]), torch.tensor([0, 1]), 8, 4, -1)
    assert ok == (0, -1)
    cases = [
        ([0, 6, 5], [0, 1], 1),
        ([-1, 2, 5], [0, 1], 0),
        ([0, 2, 9], [0, 1], 2),
        ([0, 2, 5], [0, 4], 1),
        ([0, 2, 5], [-2, 1], 0),
        ([0, 2, 5], [1, 1], 1),
    ]
    for qsl, ci, bad in cases:
        st, where = kda.validate_metadata(torch.tensor(qsl), torch.tensor(ci), 8, 4, -1)
        assert st == kda.KDA_ERR_METADATA and where == bad, (qsl, ci, st, where)
    assert kda.validate_metadata(torch.tensor([0, 2, 5]), torch.tensor([-1, -1]), 8, 4, -1)[0] == 0


def _layout(kda, dtype=0, width=3, sstride=(3 * 4608, 3, 1), wstride=(4, 1), sdtype=2,
            reserved=0):
    lay = kda.make_layout(dtype, width, sstride, wstride, sdtype)
    lay.reserved = reserved
    return lay


@pytest.mark.parametrize("lay,over,status", [
    ({}, {}, 0),
    ({"dtype": 1}, {}, 0),
    ({"dtype": 2}, {}, 0),
    ({"dtype": 3}, {}, 1),
    ({"width": 2}, {}, 1),
    ({"width": 65}, {}, 2),
    ({"width": 8, "sstride": (8, 8 * 100000, 1)}, {}, 0),
    ({"dtype": 2}, {"x_row_stride": 6404}, 0),  # fp32 rows: 16 bytes = 4 elements
    ({"dtype": 1}, {"x_row_stride": 6404}, 3),  # fp16 rows: 8 elements
    ({"wstride": (1, 4608)}, {"weight": A16 + 4}, 0),  # strided weight: 4-byte alignment
    ({}, {"weight": A16 + 4}, 3),  # dense weight: 16-byte alignment
    ({"sstride": (3 * 4608, 1, 4608)}, {"conv_states": A16 + 4}, 0),
    ({}, {"conv_states": A16 + 4}, 3),
    ({"sstride": (3 * 4608, 1, 4608)}, {"conv_states": A16 + 2}, 3),
    ({"sdtype": 0}, {}, 0),  # bf16 conv state
    ({"sdtype": 1}, {}, 1),  # fp16 conv state: not offered
    ({"sdtype": 3}, {}, 1),
    ({"reserved": 1}, {}, 1),
    ({"sdtype": 0}, {"conv_states": A16 + 8}, 3),  # dense bf16 state: 16-byte alignment
    ({"sdtype": 0, "sstride": (3 * 4608, 1, 4608)}, {"conv_states": A16 + 2}, 0),
    ({"sdtype": 0, "width": 4, "sstride": (4 * 4608, 4, 1)}, {"conv_states": A16 + 2}, 0),
])
def test_layout_checks(kda, lay, over, status):
    a = good_args(**over)
    st = kda.check_args_ex(a["x"], a["x_row_stride"], a["tokens"], a["dim"], a["part_dim"],
                           a["weight"], a["bias"], a["conv_states"], a["cache_indices"],
                           a["has_initial_state"], a["query_start_loc"], a["num_seqs"],
                           a["activation"], a["out"], _layout(kda, **lay))
    assert st == status


def test_null_layout_is_the_default(kda):
    a = good_args(weight=A16 + 4)
    args = (a["x"], a["x_row_stride"], a["tokens"], a["dim"], a["part_dim"], a["weight"],
            a["bias"], a["conv_states"], a["cache_indices"], a["has_initial_state"],
            a["query_start_loc"], a["num_seqs"], a["activation"], a["out"])
    assert kda.check_args_ex(*args, None) == kda.check_args(*args) == 3


def test_layout_struct_matches_the_header(kda):
    """kda_conv_layout_t: two int32, five int64, two int32 (56 bytes, no padding)."""
    import ctypes

    assert ctypes.sizeof(kda.KdaConvLayout) == 56
    assert kda.KdaConvLayout.state_dtype.offset == 48
    lay = kda.make_layout(0, 3, (9, 3, 1), (4, 1))
    assert lay.state_dtype == kda.KDA_DTYPE_F32 and lay.reserved == 0


def test_layout_of_maps_the_state_dtype(kda):
    x = torch.zeros(8, 128, dtype=torch.float16)
    w = torch.zeros(128, 4)
    assert kda.layout_of(x, w, torch.zeros(2, 128, 3)).state_dtype == kda.KDA_DTYPE_F32
    lay = kda.layout_of(x, w, torch.zeros(2, 128, 5, dtype=torch.bfloat16))
    assert (lay.state_dtype, lay.x_dtype, lay.state_width) == (kda.KDA_DTYPE_BF16,
                                                               kda.KDA_DTYPE_F16, 5)
    with pytest.raises(TypeError):
        kda.layout_of(x, w, torch.zeros(2, 128, 3, dtype=torch.float16))


def test_supported_predicate_rejects_host_tensors(kda):
    x = torch.zeros(8, 128, dtype=torch.bfloat16)
    w = torch.zeros(128, 4)
    st = torch.zeros(2, 128, 3)
    assert not kda.packed_causal_conv1d_supported(x, w, st, 64)


@pytest.mark.parametrize("mask,head_dim,eps,dim,part_dim,status", [
    (0b011, 128, 1e-6, 4608, 1536, 0),
    (0b011, 64, 1e-6, 3264, 1088, 0),
    (0b011, 128, 1e-6, 3264, 1088, 2),  # 1088 is not a multiple of 128
    (0b111, 4, 0.0, 4608, 1536, 0),
    (0b1000, 128, 1e-6, 4608, 1536, 1),  # plane 3 of 3
    (0b011, 96, 1e-6, 4608, 1536, 2),  # 24 lanes: not a power of two
    (0b011, 256, 1e-6, 4608, 1536, 2),  # more than a warp
    (0b011, 2, 1e-6, 4608, 1536, 2),  # less than one lane's channels
    (0b011, 128, -1e-6, 4608, 1536, 1),
    (0b011, 128, float("nan"), 4608, 1536, 1),
    (0b011, 128, float("inf"), 4608, 1536, 1),
    (0, 7, -5.0, 4608, 1536, 0),  # empty mask: no norm, nothing else checked
])
def test_l2norm_checks(kda, mask, head_dim, eps, dim, part_dim, status):
    assert kda.l2norm_check(kda.make_l2norm(mask, head_dim, eps), dim, part_dim) == status


def test_l2norm_reserved_and_null(kda):
    norm = kda.make_l2norm(0b011, 128, 1e-6)
    norm.reserved = 1
    assert kda.l2norm_check(norm, 4608, 1536) == 1
    assert kda.l2norm_check(None, 4608, 1536) == 0
    assert kda.l2norm_check(kda.make_l2norm(1, 64, 0.0), 4608, 0) == 1  # bad sizes first


def test_l2norm_struct_matches_the_header(kda):
    import ctypes

    assert ctypes.sizeof(kda.KdaL2Norm) == 16
    assert kda.KdaL2Norm.eps.offset == 8
