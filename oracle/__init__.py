"""CPU oracle for the packed varlen causal depthwise conv1d (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg and reference (oracle) arm may import this package.  The product path (the CUDA library and
its Python binding) never touches it, and it never touches the product path.

The arithmetic lives in ``kda_conv_ref.c`` (plain single-threaded C, FP32 as
the vLLM page "vllm.models.kimi_k3.nvidia.ops.kda_conv" fixes it: module
docstring, 3rd and 4th paragraphs, and the packed_causal_conv1d_fn docstring).
This module compiles it with gcc and marshals numpy arrays into it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_conv_ref.c")
_LIB_PATH = os.path.join(_HERE, "libkda_conv_ref.so")
_lock = threading.Lock()
_lib = None

REF_OK = 0
REF_BAD_SHAPE = 1
REF_BAD_QSL = 2
REF_BAD_CACHE_INDEX = 3
REF_DUP_CACHE_INDEX = 4

# No contraction of a*b+c into FMA behind the source's back: every fused
# multiply-add in the oracle is an explicit fmaf().
CFLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compiles the oracle into a shared library and returns its path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.kda_ref_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.kda_ref_bf16_to_f32.restype = ctypes.c_float
    lib.kda_ref_bf16_rne.argtypes = [ctypes.c_float]
    lib.kda_ref_bf16_rne.restype = ctypes.c_uint16
    lib.kda_ref_silu.argtypes = [ctypes.c_float]
    lib.kda_ref_silu.restype = ctypes.c_float
    for name in ("kda_ref_bf16_to_f32_n", "kda_ref_bf16_rne_n", "kda_ref_silu_n"):
        getattr(lib, name).argtypes = [P, I64, P]
        getattr(lib, name).restype = None
    lib.kda_ref_silu_bf16_range.argtypes = [ctypes.c_uint32, ctypes.c_uint64, P]
    lib.kda_ref_silu_bf16_range.restype = None
    lib.kda_ref_check_metadata.argtypes = [I64, I64, P, P, I64, I64, ctypes.POINTER(I64)]
    lib.kda_ref_check_metadata.restype = ctypes.c_int
    lib.kda_ref_packed_conv1d.argtypes = [
        P, I64, I64, I64, I64,  # x, x_row_stride, tokens, dim, part_dim
        P, P, P, I64,  # weight, bias, conv_states, cache_lines
        P, P, P, I64, I64,  # cache_indices, has_initial_state, qsl, num_seqs, null_block_id
        ctypes.c_int, P, P, P,  # activation, out, preact, act
    ]
    lib.kda_ref_packed_conv1d.restype = ctypes.c_int
    for name in ("kda_ref_f16_to_f32_n", "kda_ref_f16_rne_n"):
        getattr(lib, name).argtypes = [P, I64, P]
        getattr(lib, name).restype = None
    lib.kda_ref_packed_conv1d_ex.argtypes = [
        P, ctypes.c_int, I64, I64, I64, I64,  # x, dtype, x_row_stride, tokens, dim, part_dim
        P, I64, I64, I64, P,  # weight, w_stride_c, w_stride_j, w_stride_part, bias
        P, ctypes.c_int, I64, I64, I64, I64, I64,  # conv_states, state dtype, lines, width, strides
        P, P, P, I64, I64,  # cache_indices, has_initial_state, qsl, num_seqs, null_block_id
        ctypes.c_int, P, P,  # activation, out, preact
    ]
    lib.kda_ref_packed_conv1d_ex.restype = ctypes.c_int
    lib.kda_ref_l2norm_heads.argtypes = [P, I64, I64, I64, ctypes.c_double, P]
    lib.kda_ref_l2norm_heads.restype = ctypes.c_int
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Returns the oracle library, building it on first use."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _ptr(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def bf16_to_f32(bits: np.ndarray, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Widens bf16 bit patterns (uint16) to fp32, elementwise, via the oracle."""
    lib = lib or load()
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    out = np.empty(flat.size, dtype=np.float32)
    lib.kda_ref_bf16_to_f32_n(flat.ctypes.data, flat.size, out.ctypes.data)
    return out.reshape(np.shape(bits))


def bf16_rne(values: np.ndarray, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Rounds fp32 values to bf16 bit patterns (uint16), elementwise, via the oracle."""
    lib = lib or load()
    flat = np.ascontiguousarray(values, dtype=np.float32).ravel()
    out = np.empty(flat.size, dtype=np.uint16)
    lib.kda_ref_bf16_rne_n(flat.ctypes.data, flat.size, out.ctypes.data)
    return out.reshape(np.shape(values))


def silu(values: np.ndarray, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """SiLU in fp32, elementwise, via the oracle."""
    lib = lib or load()
    flat = np.ascontiguousarray(values, dtype=np.float32).ravel()
    out = np.empty(flat.size, dtype=np.float32)
    lib.kda_ref_silu_n(flat.ctypes.data, flat.size, out.ctypes.data)
    return out.reshape(np.shape(values))


def silu_bf16_range(first: int, count: int, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """bf16_rne(silu(f)) for the fp32 bit patterns first .. first+count-1."""
    lib = lib or load()
    out = np.empty(count, dtype=np.uint16)
    lib.kda_ref_silu_bf16_range(first, count, out.ctypes.data)
    return out


def check_metadata(tokens, cache_lines, cache_indices, query_start_loc, null_block_id,
                   lib: ctypes.CDLL | None = None) -> tuple[int, int]:
    """(status, offending sequence index or -1) for one call's metadata."""
    lib = lib or load()
    ci = np.ascontiguousarray(cache_indices, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    bad = ctypes.c_int64(-1)
    rc = lib.kda_ref_check_metadata(tokens, cache_lines, _ptr(ci), _ptr(qsl), qsl.size - 1,
                                    null_block_id, ctypes.byref(bad))
    return rc, bad.value


def packed_conv1d(x_bits: np.ndarray, col_offset: int, dim: int, part_dim: int,
                  weight: np.ndarray,
                  bias: np.ndarray | None, conv_states: np.ndarray, cache_indices: np.ndarray,
                  has_initial_state: np.ndarray, query_start_loc: np.ndarray,
                  null_block_id: int, activation: int, out: np.ndarray | None = None,
                  want_preact: bool = False, want_act: bool = False,
                  lib: ctypes.CDLL | None = None) -> dict:
    """Runs the oracle conv.

    ``x_bits`` is a (tokens, row_stride) uint16 array of bf16 bits (the whole
    in_proj buffer); the input is its columns [col_offset, col_offset + dim).
    ``conv_states`` (cache_lines, dim, 3) float32 is updated in place.  ``out``
    (dim/part_dim, tokens, part_dim) uint16, if given, is written in place
    (rows outside the sequences keep their contents); otherwise a fresh array
    filled with 0xFFFF is used.  Returns a dict with ``out`` and, on request,
    ``preact`` / ``act`` (float32, same layout, NaN where not written).
    """
    lib = lib or load()
    assert x_bits.dtype == np.uint16 and x_bits.ndim == 2
    assert x_bits.flags["C_CONTIGUOUS"]
    tokens, row_stride = x_bits.shape
    assert 0 <= col_offset and col_offset + dim <= row_stride
    assert conv_states.dtype == np.float32 and conv_states.flags["C_CONTIGUOUS"]
    assert conv_states.ndim == 3 and conv_states.shape[1:] == (dim, 3)
    weight = np.ascontiguousarray(weight, dtype=np.float32)
    bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    ci = np.ascontiguousarray(cache_indices, dtype=np.int32)
    his = np.ascontiguousarray(has_initial_state, dtype=np.uint8)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    num_seqs = qsl.size - 1
    planes = dim // part_dim if part_dim > 0 else 0
    if out is None:
        out = np.full((planes, tokens, part_dim), 0xFFFF, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.flags["C_CONTIGUOUS"]
    preact = np.full(out.shape, np.nan, dtype=np.float32) if want_preact else None
    act = np.full(out.shape, np.nan, dtype=np.float32) if want_act else None
    rc = lib.kda_ref_packed_conv1d(
        x_bits.ctypes.data + 2 * col_offset, row_stride, tokens, dim, part_dim,
        _ptr(weight), _ptr(bias), _ptr(conv_states), conv_states.shape[0],
        _ptr(ci), _ptr(his), _ptr(qsl), num_seqs, null_block_id,
        activation, _ptr(out), _ptr(preact), _ptr(act))
    if rc != REF_OK:
        raise ValueError(f"oracle rejected the call: status {rc}")
    res = {"out": out}
    if want_preact:
        res["preact"] = preact
    if want_act:
        res["act"] = act
    return res


DTYPE_BF16, DTYPE_F16, DTYPE_F32 = 0, 1, 2


def f16_to_f32(bits: np.ndarray, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Widens IEEE binary16 bit patterns (uint16) to fp32 via the oracle."""
    lib = lib or load()
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    out = np.empty(flat.size, dtype=np.float32)
    lib.kda_ref_f16_to_f32_n(flat.ctypes.data, flat.size, out.ctypes.data)
    return out.reshape(np.shape(bits))


def f16_rne(values: np.ndarray, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Rounds fp32 values to binary16 bit patterns (uint16) via the oracle."""
    lib = lib or load()
    flat = np.ascontiguousarray(values, dtype=np.float32).ravel()
    out = np.empty(flat.size, dtype=np.uint16)
    lib.kda_ref_f16_rne_n(flat.ctypes.data, flat.size, out.ctypes.data)
    return out.reshape(np.shape(values))


def _elem_strides(a: np.ndarray) -> list[int]:
    assert all(st % a.itemsize == 0 for st in a.strides)
    return [st // a.itemsize for st in a.strides]


def packed_conv1d_ex(x_buf: np.ndarray, dtype: int, col_offset: int, dim: int, part_dim: int,
                     weight: np.ndarray, bias: np.ndarray | None, conv_states: np.ndarray,
                     cache_indices, has_initial_state, query_start_loc, null_block_id: int,
                     activation: int, want_preact: bool = False,
                     lib: ctypes.CDLL | None = None) -> dict:
    """The general-layout oracle conv.

    ``x_buf`` (tokens, row_stride): uint16 bits for bf16 / fp16, float32 for
    fp32; the input is columns [col_offset, col_offset + dim).  ``weight`` is
    a (dim, 4) float32 view with any strides, or a (dim / part_dim, 4,
    part_dim) view (part, tap, channel within the part: the width-major
    decode weight of the kda_decode page) with any strides; ``conv_states`` a
    (lines, dim, K) view with any strides, float32 or uint16 (bf16 bits),
    updated in place.  Returns
    ``out`` (dim/part_dim, tokens, part_dim) of x's storage type, filled with
    0xFFFF bits (NaN for fp32) where no sequence writes, and optionally
    ``preact``."""
    lib = lib or load()
    assert x_buf.ndim == 2 and x_buf.flags["C_CONTIGUOUS"]
    assert (x_buf.dtype == np.float32) == (dtype == DTYPE_F32)
    tokens, row_stride = x_buf.shape
    assert weight.dtype == np.float32
    if weight.ndim == 2:
        assert weight.shape == (dim, 4)
        ws = _elem_strides(weight)
        w_c, w_j, w_part = ws[0], ws[1], part_dim * ws[0]
    else:
        assert weight.shape == (dim // part_dim, 4, part_dim)
        ws = _elem_strides(weight)
        w_c, w_j, w_part = ws[2], ws[1], ws[0]
    assert conv_states.dtype in (np.float32, np.uint16) and conv_states.ndim == 3
    state_dtype = DTYPE_F32 if conv_states.dtype == np.float32 else DTYPE_BF16
    assert conv_states.shape[1] == dim
    ss = _elem_strides(conv_states)
    bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    ci = np.ascontiguousarray(cache_indices, dtype=np.int32)
    his = np.ascontiguousarray(has_initial_state, dtype=np.uint8)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    planes = dim // part_dim
    if dtype == DTYPE_F32:
        out = np.full((planes, tokens, part_dim), np.nan, dtype=np.float32)
    else:
        out = np.full((planes, tokens, part_dim), 0xFFFF, dtype=np.uint16)
    preact = np.full(out.shape, np.nan, dtype=np.float32) if want_preact else None
    rc = lib.kda_ref_packed_conv1d_ex(
        x_buf.ctypes.data + x_buf.itemsize * col_offset, dtype, row_stride, tokens, dim, part_dim,
        weight.ctypes.data, w_c, w_j, w_part, _ptr(bias),
        conv_states.ctypes.data, state_dtype, conv_states.shape[0], conv_states.shape[2],
        ss[0], ss[1], ss[2],
        _ptr(ci), _ptr(his), _ptr(qsl), qsl.size - 1, null_block_id, activation,
        out.ctypes.data, _ptr(preact))
    if rc != REF_OK:
        raise ValueError(f"oracle rejected the call: status {rc}")
    res = {"out": out}
    if want_preact:
        res["preact"] = preact
    return res


def l2norm_heads(y: np.ndarray, head_dim: int, eps: float,
                 lib: ctypes.CDLL | None = None) -> np.ndarray:
    """The per-head L2 norm of (rows, width) fp32 values, in float64."""
    lib = lib or load()
    y = np.ascontiguousarray(y, dtype=np.float32)
    assert y.ndim == 2
    out = np.empty(y.shape, dtype=np.float64)
    rc = lib.kda_ref_l2norm_heads(y.ctypes.data, y.shape[0], y.shape[1], head_dim, float(eps),
                                  out.ctypes.data)
    if rc != REF_OK:
        raise ValueError(f"oracle rejected the call: status {rc}")
    return out


def packed_conv1d_l2norm(x_buf: np.ndarray, dtype: int, col_offset: int, dim: int,
                         part_dim: int, weight: np.ndarray, bias: np.ndarray | None,
                         conv_states: np.ndarray, cache_indices, has_initial_state,
                         query_start_loc, null_block_id: int, activation: int,
                         norm_planes: int, head_dim: int, eps: float,
                         lib: ctypes.CDLL | None = None) -> dict:
    """The conv with the q/k L2 norm folded in: the planes whose bit is set in
    ``norm_planes`` hold each token's heads divided by their L2 norm.

    Steps, each an oracle function: the general-layout conv (its FP32
    pre-activations; the conv state is updated as by packed_conv1d_ex), the
    FP32 activation, the per-head norm in float64, rounding to float32 and then
    to x's storage type.  Planes outside the mask are the plain conv output.
    Returns ``out`` as packed_conv1d_ex does."""
    lib = lib or load()
    res = packed_conv1d_ex(x_buf, dtype, col_offset, dim, part_dim, weight, bias, conv_states,
                           cache_indices, has_initial_state, query_start_loc, null_block_id,
                           activation, want_preact=True, lib=lib)
    pre = res["preact"]
    out = res["out"]
    post = silu(pre, lib) if activation else pre
    for plane in range(dim // part_dim):
        if not (norm_planes >> plane) & 1:
            continue
        rows = ~np.isnan(pre[plane][:, 0])  # token rows some sequence wrote
        normed = l2norm_heads(post[plane][rows], head_dim, eps, lib).astype(np.float32)
        if dtype == DTYPE_BF16:
            out[plane][rows] = bf16_rne(normed, lib)
        elif dtype == DTYPE_F16:
            out[plane][rows] = f16_rne(normed, lib)
        else:
            out[plane][rows] = normed
    return {"out": out}
