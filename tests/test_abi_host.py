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
            version=1, wpart=0, ci_stride=0):
    lay = kda.make_layout(dtype, width, sstride, wstride, sdtype, wpart, ci_stride)
    lay.version = version
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
    ({"version": 2}, {}, 1),
    ({"version": -1}, {}, 1),
    ({"version": 0, "ci_stride": -5}, {}, 0),  # version 0: the version-1 fields are not read
    ({"ci_stride": -1}, {}, 1),
    ({"ci_stride": 3}, {}, 0),
    # the kda_decode page's [qkv, width, channel] weight: strided, 4-byte alignment
    ({"wstride": (1, 1536), "wpart": 4 * 1536}, {"weight": A16 + 4}, 0),
    # (4, 1) with the part stride of one (dim, 4) array is dense: 16-byte alignment
    ({"wpart": 4 * 1536}, {"weight": A16 + 4}, 3),
    # (4, 1) with a padded part stride is not one array: 4-byte alignment
    ({"wpart": 4 * 1536 + 4}, {"weight": A16 + 4}, 0),
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

    assert ctypes.sizeof(kda.KdaConvLayout) == 72
    assert kda.KdaConvLayout.state_dtype.offset == 48
    assert kda.KdaConvLayout.version.offset == 52
    assert kda.KdaConvLayout.weight_part_stride.offset == 56
    assert kda.KdaConvLayout.cache_index_stride.offset == 64
    lay = kda.make_layout(0, 3, (9, 3, 1), (4, 1))
    assert lay.state_dtype == kda.KDA_DTYPE_F32 and lay.version == 1
    assert lay.weight_part_stride == 0 and lay.cache_index_stride == 0


def test_version0_layout_is_read_as_the_shorter_struct(kda):
    """A caller built against the 56-byte struct (version 0, no part or
    cache-index stride) is read without touching the bytes after it: the
    struct is placed at the very end of a page-sized buffer's used part, and
    whatever follows it (here: a poison pattern) is ignored."""
    import ctypes

    class Old(ctypes.Structure):
        _fields_ = [("x_dtype", ctypes.c_int32), ("state_width", ctypes.c_int32),
                    ("state_stride", ctypes.c_int64 * 3), ("weight_stride", ctypes.c_int64 * 2),
                    ("state_dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]

    buf = (ctypes.c_uint8 * 72)(*([0] * 56 + [0xFF] * 16))  # poison after the old struct
    old = Old.from_buffer(buf)
    old.x_dtype, old.state_width, old.state_dtype, old.reserved = 0, 3, 2, 0
    old.state_stride[:] = (3 * 4608, 3, 1)
    old.weight_stride[:] = (4, 1)
    a = good_args()
    st = kda.check_args_ex(a["x"], a["x_row_stride"], a["tokens"], a["dim"], a["part_dim"],
                           a["weight"], a["bias"], a["conv_states"], a["cache_indices"],
                           a["has_initial_state"], a["query_start_loc"], a["num_seqs"],
                           a["activation"], a["out"],
                           ctypes.cast(ctypes.pointer(old), ctypes.POINTER(kda.KdaConvLayout)).contents)
    assert st == 0  # a poisoned cache-index stride (-1) would be rejected


def test_layout_of_reads_the_decode_weight_and_index_strides(kda):
    x = torch.zeros(8, 192, dtype=torch.bfloat16)
    w3 = torch.zeros(3, 4, 64)  # [qkv, width, channel]
    ci = torch.zeros(10, dtype=torch.int32)[::2]
    lay = kda.layout_of(x, w3, torch.zeros(2, 192, 3), ci)
    assert tuple(lay.weight_stride) == (1, 64) and lay.weight_part_stride == 256
    assert lay.cache_index_stride == 2 and lay.version == 1
    lay = kda.layout_of(x, torch.zeros(192, 4), torch.zeros(2, 192, 3))
    assert tuple(lay.weight_stride) == (4, 1) and lay.weight_part_stride == 0


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
    (0b011, 128, 1e-40, 4608, 1536, 1),  # subnormal: flushed by the SFU root
    (0b011, 128, 1.1754944e-38, 4608, 1536, 0),  # FLT_MIN
    (0b011, 128, 1e-30, 4608, 1536, 0),
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


def test_window_search_model(kda):
    """Host model of the device's one-round window search: for every program
    p, the owner s (the largest s with f(s) = floor(qsl[s] / chunk) + s <= p)
    lies in [p - ceil(tokens / chunk), p], the entry after it is inside the
    loaded window [lo, min(num_seqs, p + 1)], which holds at most
    ceil(tokens / chunk) + 2 entries, and counting the window's candidates j
    that pass q < (p - j + 1) * chunk finds s."""
    rng = np.random.default_rng(11)
    for trial in range(150):
        n = int(rng.integers(1, 400))
        kind = trial % 3
        if kind == 0:
            lens = rng.integers(0, 300, size=n)
        elif kind == 1:
            lens = rng.integers(0, 3, size=n)
        else:
            lens = np.where(rng.random(n) < 0.02, rng.integers(1000, 9000, size=n),
                            rng.integers(0, 40, size=n))
        qsl = np.concatenate([[int(rng.integers(0, 50))], lens]).cumsum()
        tokens = int(qsl[-1] + rng.integers(0, 20))
        sh = kda.launch_shape(tokens, 4608, 1536, n)
        chunk, programs = sh["chunk"], sh["programs"]
        span = -(-tokens // chunk)
        f = qsl[:-1] // chunk + np.arange(n)
        p = np.arange(programs)
        s = np.searchsorted(f, p, side="right") - 1  # owner, -1 before the first
        lo, hi = np.maximum(0, p - span), np.minimum(n, p + 1)
        assert (hi - lo + 1 <= span + 2).all()
        own = s >= 0
        assert ((lo <= s) & (s < hi))[own].all(), trial
        # the counted candidates: j in [lo, hi) with q < (p - j + 1) * chunk
        for pi in rng.choice(programs, size=min(programs, 40), replace=False):
            j = np.arange(lo[pi], hi[pi])
            ok = qsl[j] < (pi - j + 1) * chunk
            assert (ok == (f[j] <= pi)).all()
            assert int(ok.sum()) - 1 + lo[pi] == s[pi] or (s[pi] == -1 and not ok.any())


def test_chunk_bounded_for_many_sequences(kda):
    """The chunk stays near the even spread of the tokens over the resident
    warps whatever the sequence count: with 2..117 sequences at 16K tokens
    (3 x 1536 channels: 36 warps per program, 118 programs per wave of
    152 x 7 CTAs) it is the two-wave spread, 72 rows, where the one-wave fit
    alone would give up to 2048 rows (one long prompt among short ones then
    streams through a few warps); one sequence keeps the one-wave fit (144
    rows) and 118 or more take the one-wave spread."""
    spread2 = -(-16384 * 36 // (2 * 152 * 4 * 7))
    assert kda.launch_shape(16384, 4608, 1536, 1)["chunk"] == 144
    for n in range(2, 118):
        sh = kda.launch_shape(16384, 4608, 1536, n)
        assert sh["chunk"] == -(-spread2 // 6) * 6 == 72, n
    for n in (118, 200, 1280):
        assert kda.launch_shape(16384, 4608, 1536, n)["chunk"] == -(-16384 * 36 // 4256 // 6) * 6
    # small batches keep the one-wave fit (no less than 48 rows from the cap)
    assert kda.launch_shape(2430, 4608, 1536, 8)["chunk"] == 24
    assert kda.launch_shape(2600, 4608, 1536, 31)["chunk"] == 30


def test_fast_division_model():
    """Host model of the kernel's division by a launch-fixed divisor (chunk,
    warps per program): with l = ceil(log2 d), m = floor(2^32 (2^l - d) / d)
    + 1, t = umulhi(m, n), the quotient (t + ((n - t) >> min(l, 1))) >>
    max(l - 1, 0) equals n // d for every 32-bit n, checked for d = 1..4096,
    powers of two and their neighbours up to 2^30, and random d, against
    edge and random numerators."""
    rng = np.random.default_rng(17)
    ds = list(range(1, 4097)) + [2 ** k + o for k in range(12, 31) for o in (-1, 0, 1)]
    ds += [int(v) for v in rng.integers(1, 2 ** 31, size=300)]
    for d in ds:
        l = 0
        while (1 << l) < d:
            l += 1
        m = ((1 << 32) * ((1 << l) - d)) // d + 1
        assert 0 < m < (1 << 32)
        s1, s2 = min(l, 1), max(l - 1, 0)
        n = np.concatenate([np.array([0, 1, d - 1, d, d + 1, 2 * d - 1, 2 * d, 2 ** 32 - 1,
                                      2 ** 31, (2 ** 32 - 1) // d * d], dtype=np.uint64),
                            rng.integers(0, 2 ** 32, size=200, dtype=np.uint64)])
        n = n[n < 2 ** 32]
        t = (np.uint64(m) * n) >> np.uint64(32)
        q = (t + ((n - t) >> np.uint64(s1))) >> np.uint64(s2)
        assert np.array_equal(q, n // np.uint64(d)), d


def test_index_range_limits(kda):
    """Launch sizes whose device-side 32-bit index division would overflow
    are rejected before any CUDA call: a decode update of 2^34 (token,
    vector) items, and a packed launch of more than 2^32 warps."""
    with pytest.raises(kda.KdaError) as e:
        kda.kda_conv1d_update(A16, 4096, 1 << 24, 4096, 1024, A16, A16, A16, A16, -1, 1, A16,
                              None, stream=0)
    assert e.value.status == kda.KDA_ERR_INVALID_ARG
    with pytest.raises(kda.KdaError) as e:
        kda.kda_packed_conv1d(A16, 1 << 24, (1 << 31) - 1, 1 << 24, 1 << 22, A16, A16, A16, A16,
                              A16, A16, 1, -1, 1, A16, stream=0)
    assert e.value.status == kda.KDA_ERR_INVALID_ARG
