"""ctypes marshalling for libkdaconv.so (argument conversion only)."""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_MISALIGNED = 3
KDA_ERR_CUDA = 4
KDA_ERR_METADATA = 5
KDA_ACT_NONE = 0
KDA_ACT_SILU = 1
KDA_DTYPE_BF16 = 0
KDA_DTYPE_F16 = 1
KDA_DTYPE_F32 = 2

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    """A non-zero kda_status_t from the library."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(what)


class KdaConvLayout(ctypes.Structure):
    """kda_conv_layout_t (version 1): x/out dtype, conv-state width, element
    strides, conv-state dtype, the weight's part stride and the stride of
    cache_indices."""

    _fields_ = [("x_dtype", ctypes.c_int32), ("state_width", ctypes.c_int32),
                ("state_stride", ctypes.c_int64 * 3), ("weight_stride", ctypes.c_int64 * 2),
                ("state_dtype", ctypes.c_int32), ("version", ctypes.c_int32),
                ("weight_part_stride", ctypes.c_int64), ("cache_index_stride", ctypes.c_int64)]


def make_layout(x_dtype: int, state_width: int, state_stride, weight_stride,
                state_dtype: int = KDA_DTYPE_F32, weight_part_stride: int = 0,
                cache_index_stride: int = 0) -> KdaConvLayout:
    """A version-1 layout; weight_part_stride 0 = one (dim, 4) weight array,
    cache_index_stride 0 = contiguous cache indices."""
    return KdaConvLayout(x_dtype, state_width, (ctypes.c_int64 * 3)(*state_stride),
                         (ctypes.c_int64 * 2)(*weight_stride), state_dtype, 1,
                         weight_part_stride, cache_index_stride)


class KdaL2Norm(ctypes.Structure):
    """kda_l2norm_t: planes to normalise per head, head size, epsilon."""

    _fields_ = [("plane_mask", ctypes.c_uint32), ("head_dim", ctypes.c_int32),
                ("eps", ctypes.c_float), ("reserved", ctypes.c_int32)]


def make_l2norm(plane_mask: int, head_dim: int = 128, eps: float = 1e-6) -> KdaL2Norm:
    return KdaL2Norm(plane_mask, head_dim, eps, 0)


def lib_path() -> str:
    return _build.LIB_PATH


def _declare(handle: ctypes.CDLL) -> ctypes.CDLL:
    P, I64, I32, C = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
    conv = [P, I64, I64, I64, I64, P, P, P, P, P, P, I64, I64]
    handle.kda_packed_conv1d.argtypes = conv + [C, P, P]
    handle.kda_packed_conv1d_preact_f32.argtypes = conv + [P, P]
    handle.kda_packed_conv1d_ex.argtypes = conv + [C, P, ctypes.POINTER(KdaConvLayout), P]
    handle.kda_conv1d_update.argtypes = [P, I64, I64, I64, I64, P, P, P, P, I64, C, P,
                                         ctypes.POINTER(KdaConvLayout), P]
    handle.kda_packed_conv1d_l2norm.argtypes = conv + [C, P, ctypes.POINTER(KdaConvLayout),
                                                       ctypes.POINTER(KdaL2Norm), P]
    handle.kda_conv1d_update_l2norm.argtypes = [P, I64, I64, I64, I64, P, P, P, P, I64, C, P,
                                                ctypes.POINTER(KdaConvLayout),
                                                ctypes.POINTER(KdaL2Norm), P]
    handle.kda_l2norm_check.argtypes = [ctypes.POINTER(KdaL2Norm), I64, I64]
    handle.kda_packed_conv1d_ex_check_args.argtypes = [P, I64, I64, I64, I64, P, P, P, P, P, P,
                                                       I64, C, P, ctypes.POINTER(KdaConvLayout)]
    handle.kda_packed_conv1d_check_args.argtypes = [P, I64, I64, I64, I64, P, P, P, P, P, P, I64,
                                                    C, P]
    handle.kda_packed_conv1d_launch_shape.argtypes = [
        I64, I64, I64, I64, I32, ctypes.POINTER(I64), ctypes.POINTER(I32), ctypes.POINTER(I32),
        ctypes.POINTER(I64)]
    handle.kda_validate_metadata.argtypes = [P, P, I64, I64, I64, I64, ctypes.POINTER(I64)]
    handle.kda_validate_metadata_device.argtypes = [P, P, I64, I64, I64, I64, I64,
                                                    ctypes.POINTER(I64), P]
    handle.kda_validate_metadata_device_noalloc.argtypes = [P, P, I64, I64, I64, I64, I64,
                                                            ctypes.POINTER(I64), P]
    handle.kda_epilogue_range.argtypes = [ctypes.c_uint32, ctypes.c_uint64, C, P, P]
    for name in ("kda_packed_conv1d", "kda_packed_conv1d_preact_f32", "kda_packed_conv1d_ex",
                 "kda_conv1d_update", "kda_packed_conv1d_l2norm", "kda_conv1d_update_l2norm",
                 "kda_l2norm_check",
                 "kda_packed_conv1d_ex_check_args",
                 "kda_packed_conv1d_check_args", "kda_packed_conv1d_launch_shape",
                 "kda_validate_metadata", "kda_validate_metadata_device",
                 "kda_validate_metadata_device_noalloc", "kda_epilogue_range"):
        getattr(handle, name).restype = C
    handle.kda_status_string.argtypes = [C]
    handle.kda_status_string.restype = ctypes.c_char_p
    handle.kda_last_error_string.argtypes = []
    handle.kda_last_error_string.restype = ctypes.c_char_p
    return handle


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built: there is no fallback."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it first (linear_attention_prefill_varlen_gb300."
                    "_build.build(), or __graft_entry__.build()); there is no CPU fallback")
            _lib = _declare(ctypes.CDLL(path))
    return _lib


def _check(status: int) -> None:
    if status != KDA_OK:
        h = lib()
        what = h.kda_status_string(status).decode()
        if status == KDA_ERR_CUDA:
            what += ": " + h.kda_last_error_string().decode()
        raise KdaError(status, what)


def _ptr(t) -> int | None:
    """Device (or host) address of a tensor, an int address, or None."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def kda_packed_conv1d(x, x_row_stride: int, tokens: int, dim: int, part_dim: int, weight, bias,
                      conv_states, cache_indices, has_initial_state, query_start_loc,
                      num_seqs: int, null_block_id: int, activation: int, out,
                      stream=None) -> None:
    """C-ABI kda_packed_conv1d.  Tensors (or raw device addresses) are passed
    by pointer exactly as given; the call is asynchronous on `stream`
    (default: torch's current stream)."""
    _check(lib().kda_packed_conv1d(
        _ptr(x), x_row_stride, tokens, dim, part_dim, _ptr(weight), _ptr(bias),
        _ptr(conv_states), _ptr(cache_indices), _ptr(has_initial_state), _ptr(query_start_loc),
        num_seqs, null_block_id, activation, _ptr(out), _stream(stream)))


def kda_packed_conv1d_ex(x, x_row_stride: int, tokens: int, dim: int, part_dim: int, weight,
                         bias, conv_states, cache_indices, has_initial_state, query_start_loc,
                         num_seqs: int, null_block_id: int, activation: int, out,
                         layout: KdaConvLayout | None, stream=None) -> None:
    """C-ABI kda_packed_conv1d_ex (layout None: the default layout)."""
    _check(lib().kda_packed_conv1d_ex(
        _ptr(x), x_row_stride, tokens, dim, part_dim, _ptr(weight), _ptr(bias),
        _ptr(conv_states), _ptr(cache_indices), _ptr(has_initial_state), _ptr(query_start_loc),
        num_seqs, null_block_id, activation, _ptr(out),
        None if layout is None else ctypes.byref(layout), _stream(stream)))


def kda_conv1d_update(x, x_row_stride: int, batch: int, dim: int, part_dim: int, weight, bias,
                      conv_states, cache_indices, null_block_id: int, activation: int, out,
                      layout: KdaConvLayout | None = None, stream=None) -> None:
    """C-ABI kda_conv1d_update: one new token per sequence (decode)."""
    _check(lib().kda_conv1d_update(
        _ptr(x), x_row_stride, batch, dim, part_dim, _ptr(weight), _ptr(bias), _ptr(conv_states),
        _ptr(cache_indices), null_block_id, activation, _ptr(out),
        None if layout is None else ctypes.byref(layout), _stream(stream)))


def _byref(s):
    return None if s is None else ctypes.byref(s)


def kda_packed_conv1d_l2norm(x, x_row_stride: int, tokens: int, dim: int, part_dim: int,
                             weight, bias, conv_states, cache_indices, has_initial_state,
                             query_start_loc, num_seqs: int, null_block_id: int,
                             activation: int, out, layout: KdaConvLayout | None,
                             norm: KdaL2Norm | None, stream=None) -> None:
    """C-ABI kda_packed_conv1d_l2norm (norm None: kda_packed_conv1d_ex)."""
    _check(lib().kda_packed_conv1d_l2norm(
        _ptr(x), x_row_stride, tokens, dim, part_dim, _ptr(weight), _ptr(bias),
        _ptr(conv_states), _ptr(cache_indices), _ptr(has_initial_state), _ptr(query_start_loc),
        num_seqs, null_block_id, activation, _ptr(out), _byref(layout), _byref(norm),
        _stream(stream)))


def kda_conv1d_update_l2norm(x, x_row_stride: int, batch: int, dim: int, part_dim: int,
                             weight, bias, conv_states, cache_indices, null_block_id: int,
                             activation: int, out, layout: KdaConvLayout | None,
                             norm: KdaL2Norm | None, stream=None) -> None:
    """C-ABI kda_conv1d_update_l2norm (norm None: kda_conv1d_update)."""
    _check(lib().kda_conv1d_update_l2norm(
        _ptr(x), x_row_stride, batch, dim, part_dim, _ptr(weight), _ptr(bias), _ptr(conv_states),
        _ptr(cache_indices), null_block_id, activation, _ptr(out), _byref(layout), _byref(norm),
        _stream(stream)))


def l2norm_check(norm: KdaL2Norm | None, dim: int, part_dim: int) -> int:
    """Host-only status of these norm options (no CUDA call)."""
    return lib().kda_l2norm_check(_byref(norm), dim, part_dim)


def causal_conv1d_update(x: torch.Tensor, conv_states: torch.Tensor, weight: torch.Tensor,
                         bias: torch.Tensor | None, cache_indices: torch.Tensor, part_dim: int,
                         activation="silu", null_block_id: int | None = None,
                         out: torch.Tensor | None = None, stream=None,
                         use_qk_l2norm: bool = False, head_dim: int = 128,
                         l2norm_eps: float = 1e-6) -> torch.Tensor:
    """One decode step: x (batch, dim), row i the next token of the sequence at
    conv-state line cache_indices[i].  Returns (dim // part_dim, batch, part_dim)
    in x's dtype and shifts each touched line by one row, in place.  The
    weight may be (dim, 4) or the kda_decode page's (dim // part_dim, 4,
    part_dim) [qkv, width, channel] form, with any strides; cache_indices may
    be a strided 1-D view.  `use_qk_l2norm` as for packed_causal_conv1d_fn."""
    act = activation_code(activation)
    _check_conv_tensors(x, weight, bias, conv_states, out, part_dim, x.size(0) if x.dim() else 0)
    batch, dim = x.shape
    _check_vector("cache_indices", cache_indices, batch, (torch.int32,), strided=True)
    _check_devices(x=x, weight=weight, bias=bias, conv_states=conv_states,
                   cache_indices=cache_indices, out=out)
    if out is None:
        out = torch.empty((dim // part_dim, batch, part_dim), dtype=x.dtype, device=x.device)
    null = -(2 ** 62) if null_block_id is None else int(null_block_id)
    norm = make_l2norm(0b011, head_dim, l2norm_eps) if use_qk_l2norm else None
    kda_conv1d_update_l2norm(x, x.stride(0), batch, dim, part_dim, weight, bias, conv_states,
                             cache_indices, null, act, out,
                             layout_of(x, weight, conv_states, cache_indices), norm, stream)
    return out


def check_args_ex(x, x_row_stride, tokens, dim, part_dim, weight, bias, conv_states,
                  cache_indices, has_initial_state, query_start_loc, num_seqs, activation, out,
                  layout: KdaConvLayout | None) -> int:
    """Host-only argument check of kda_packed_conv1d_ex; returns the status."""
    return lib().kda_packed_conv1d_ex_check_args(
        _ptr(x), x_row_stride, tokens, dim, part_dim, _ptr(weight), _ptr(bias),
        _ptr(conv_states), _ptr(cache_indices), _ptr(has_initial_state), _ptr(query_start_loc),
        num_seqs, activation, _ptr(out), None if layout is None else ctypes.byref(layout))


def kda_packed_conv1d_preact_f32(x, x_row_stride: int, tokens: int, dim: int, part_dim: int,
                                 weight, bias, conv_states, cache_indices, has_initial_state,
                                 query_start_loc, num_seqs: int, null_block_id: int, out,
                                 stream=None) -> None:
    """C-ABI kda_packed_conv1d_preact_f32: FP32 accumulators into `out`."""
    _check(lib().kda_packed_conv1d_preact_f32(
        _ptr(x), x_row_stride, tokens, dim, part_dim, _ptr(weight), _ptr(bias),
        _ptr(conv_states), _ptr(cache_indices), _ptr(has_initial_state), _ptr(query_start_loc),
        num_seqs, null_block_id, _ptr(out), _stream(stream)))


def check_args(x, x_row_stride, tokens, dim, part_dim, weight, bias, conv_states,
               cache_indices, has_initial_state, query_start_loc, num_seqs, activation,
               out) -> int:
    """Host-only argument check (never dereferences a pointer); returns the status."""
    return lib().kda_packed_conv1d_check_args(
        _ptr(x), x_row_stride, tokens, dim, part_dim, _ptr(weight), _ptr(bias),
        _ptr(conv_states), _ptr(cache_indices), _ptr(has_initial_state), _ptr(query_start_loc),
        num_seqs, activation, _ptr(out))


def launch_shape(tokens: int, dim: int, part_dim: int, num_seqs: int, sm_count: int = 152) -> dict:
    """The launch the library makes for these sizes on a GPU with `sm_count` SMs
    (0: ask the current device)."""
    ctas, programs = ctypes.c_int64(), ctypes.c_int64()
    threads, chunk = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().kda_packed_conv1d_launch_shape(tokens, dim, part_dim, num_seqs, sm_count,
                                                ctypes.byref(ctas), ctypes.byref(threads),
                                                ctypes.byref(chunk), ctypes.byref(programs)))
    return {"ctas": ctas.value, "threads": threads.value, "chunk": chunk.value,
            "programs": programs.value}


def validate_metadata(query_start_loc, cache_indices, tokens: int, cache_lines: int,
                      null_block_id: int) -> tuple[int, int]:
    """Host-side metadata check.  Accepts CPU or CUDA int32 tensors (CUDA ones
    are copied to the host, which synchronises).  Returns (status, bad seq)."""
    qsl = torch.as_tensor(query_start_loc).to("cpu", torch.int32).contiguous()
    ci = torch.as_tensor(cache_indices).to("cpu", torch.int32).contiguous()
    bad = ctypes.c_int64(-1)
    st = lib().kda_validate_metadata(qsl.data_ptr(), ci.data_ptr(), qsl.numel() - 1, tokens,
                                     cache_lines, null_block_id, ctypes.byref(bad))
    return st, bad.value


def validate_metadata_device(query_start_loc: torch.Tensor, cache_indices: torch.Tensor,
                             tokens: int, cache_lines: int, null_block_id: int,
                             stream=None, noalloc: bool = False) -> tuple[int, int]:
    """C-ABI kda_validate_metadata_device on CUDA int32 tensors (cache_indices
    may be a strided 1-D view), without copying them to the host; synchronises
    the stream.  Returns (status, bad seq) as validate_metadata does.
    noalloc=True calls kda_validate_metadata_device_noalloc instead: the same
    check on the library's fixed device scratch, for a caller that cannot
    allocate (at most 262144 cache lines; calls must not overlap)."""
    for name, t in (("query_start_loc", query_start_loc), ("cache_indices", cache_indices)):
        if t.dtype != torch.int32 or t.dim() != 1 or not t.is_cuda:
            raise ValueError(f"{name} must be a 1-D CUDA int32 tensor")
    if not query_start_loc.is_contiguous():
        raise ValueError("query_start_loc must be contiguous")
    num_seqs = max(query_start_loc.numel() - 1, 0)
    if cache_indices.numel() < num_seqs:
        raise ValueError(f"cache_indices has {cache_indices.numel()} entries, {num_seqs} needed")
    stride = cache_indices.stride(0) if cache_indices.numel() > 1 else 1
    bad = ctypes.c_int64(-1)
    fn = (lib().kda_validate_metadata_device_noalloc if noalloc
          else lib().kda_validate_metadata_device)
    st = fn(query_start_loc.data_ptr(), cache_indices.data_ptr(), stride, num_seqs, tokens,
            cache_lines, null_block_id, ctypes.byref(bad), _stream(stream))
    if st == KDA_ERR_CUDA:
        _check(st)
    return st, bad.value


def epilogue_range(first: int, count: int, activation: int, out, stream=None) -> None:
    """C-ABI kda_epilogue_range into a device uint16/int16 tensor."""
    _check(lib().kda_epilogue_range(first, count, activation, _ptr(out), _stream(stream)))


_SILU_NAMES = ("silu", "swish")
_NONE_NAMES = ("none", "identity")


def activation_code(activation) -> int:
    """The kda_activation_t of a wrapper's `activation`: "silu", "swish" or
    True select SiLU; None, False, "none" or "identity" select none.  Any
    other value (another name, a different case, an integer) is a ValueError
    rather than a silent choice."""
    if activation is True or (isinstance(activation, str) and activation in _SILU_NAMES):
        return KDA_ACT_SILU
    if activation is None or activation is False or (
            isinstance(activation, str) and activation in _NONE_NAMES):
        return KDA_ACT_NONE
    raise ValueError(f"activation must be 'silu', 'swish', True, None, False, 'none' or "
                     f"'identity', not {activation!r}")
_DTYPES = {torch.bfloat16: KDA_DTYPE_BF16, torch.float16: KDA_DTYPE_F16,
           torch.float32: KDA_DTYPE_F32}
_STATE_DTYPES = {torch.float32: KDA_DTYPE_F32, torch.bfloat16: KDA_DTYPE_BF16}


def _weight_shape_ok(weight: torch.Tensor, dim: int, part_dim: int) -> bool:
    """A (dim, 4) weight, or the kda_decode page's [qkv, width, channel] form
    (dim / part_dim, 4, part_dim); fp32, any strides."""
    if weight.dtype != torch.float32:
        return False
    if weight.dim() == 2:
        return tuple(weight.shape) == (dim, 4)
    return (weight.dim() == 3 and part_dim > 0 and dim % part_dim == 0
            and tuple(weight.shape) == (dim // part_dim, 4, part_dim))


def packed_causal_conv1d_supported(x: torch.Tensor, weight: torch.Tensor,
                                   conv_states: torch.Tensor, part_dim: int) -> bool:
    """Whether packed_causal_conv1d_fn takes these inputs: the page's predicate
    (x CUDA, 2-D, unit channel stride, bf16 / fp16 / fp32; FP32 weight (dim, 4)
    and conv_states (lines, dim, >= 3), any strides; part_dim a multiple of 64
    dividing dim) plus this library's alignment rules (x rows on 16-byte
    boundaries, state width at most 64), widened to a bf16 conv state and to
    the kda_decode page's (dim / part_dim, 4, part_dim) weight."""
    if not (x.is_cuda and x.dim() == 2 and x.stride(1) == 1 and x.dtype in _DTYPES):
        return False
    quantum = 4 if x.dtype == torch.float32 else 8
    return (
        x.stride(0) % quantum == 0 and x.data_ptr() % 16 == 0
        and _weight_shape_ok(weight, x.size(1), part_dim)
        and conv_states.dtype in _STATE_DTYPES and conv_states.dim() == 3
        and conv_states.size(1) == x.size(1) and 3 <= conv_states.size(2) <= 64
        and part_dim > 0 and part_dim % 64 == 0 and x.size(1) % part_dim == 0
    )


def _check_vector(name: str, t: torch.Tensor, need: int, dtypes: tuple,
                  strided: bool = False) -> None:
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must be {' or '.join(str(d) for d in dtypes)}, not {t.dtype}")
    if strided:
        if t.dim() != 1 or (t.numel() > 1 and t.stride(0) < 1):
            raise ValueError(f"{name} must be a 1-D tensor with a positive stride")
    elif t.dim() != 1 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 1-D tensor")
    if t.numel() < need:
        raise ValueError(f"{name} has {t.numel()} entries, {need} needed")


def _check_conv_tensors(x, weight, bias, conv_states, out, part_dim: int, rows: int) -> None:
    """Dtypes and shapes the C ABI reads the wrappers' tensors with, checked
    before any pointer reaches the library."""
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D (rows, dim) with unit channel stride")
    if x.dtype not in _DTYPES:
        raise TypeError(f"x must be bf16, fp16 or fp32, not {x.dtype}")
    dim = x.size(1)
    if not _weight_shape_ok(weight, dim, part_dim):
        raise ValueError(f"weight must be fp32 ({dim}, 4) or (parts, 4, part_dim), not "
                         f"{weight.dtype} {tuple(weight.shape)}")
    if bias is not None and (bias.dtype != torch.float32 or tuple(bias.shape) != (dim,)
                             or not bias.is_contiguous()):
        raise ValueError(f"bias must be a contiguous fp32 ({dim},) tensor or None")
    if (conv_states.dtype not in _STATE_DTYPES or conv_states.dim() != 3
            or conv_states.size(1) != dim):
        raise ValueError(f"conv_states must be fp32 or bf16 (lines, {dim}, width)")
    if part_dim <= 0 or dim % part_dim != 0:
        raise ValueError(f"part_dim {part_dim} must divide dim {dim}")
    if out is not None:
        shape = (dim // part_dim, rows, part_dim)
        if out.dtype != x.dtype or tuple(out.shape) != shape or not out.is_contiguous():
            raise ValueError(f"out must be a contiguous {x.dtype} {shape} tensor")


def _check_devices(**tensors) -> None:
    """Every tensor on x's CUDA device (there is no CPU path)."""
    dev = tensors["x"].device
    if dev.type != "cuda":
        raise ValueError("x must be a CUDA tensor: the library has no CPU path")
    for name, t in tensors.items():
        if t is not None and t.device != dev:
            raise ValueError(f"{name} is on {t.device}, x on {dev}")


def layout_of(x: torch.Tensor, weight: torch.Tensor, conv_states: torch.Tensor,
              cache_indices: torch.Tensor | None = None) -> KdaConvLayout:
    """The kda_conv_layout_t describing these tensors.  A 3-D weight is the
    (parts, 4, part_dim) [qkv, width, channel] form."""
    if conv_states.dtype not in _STATE_DTYPES:
        raise TypeError(f"conv_states must be fp32 or bf16, not {conv_states.dtype}")
    if weight.dim() == 3:
        w_stride, w_part = (weight.stride(2), weight.stride(1)), weight.stride(0)
    else:
        w_stride, w_part = weight.stride(), 0
    ci_stride = cache_indices.stride(0) if cache_indices is not None and cache_indices.numel() > 1 \
        else 0
    return make_layout(_DTYPES[x.dtype], conv_states.size(2), conv_states.stride(), w_stride,
                       _STATE_DTYPES[conv_states.dtype], w_part, ci_stride)


def packed_causal_conv1d_fn(x: torch.Tensor, weight: torch.Tensor, bias: torch.Tensor | None,
                            conv_states: torch.Tensor, query_start_loc: torch.Tensor,
                            cache_indices: torch.Tensor, has_initial_state: torch.Tensor,
                            part_dim: int, activation="silu", null_block_id: int | None = None,
                            out: torch.Tensor | None = None, stream=None,
                            use_qk_l2norm: bool = False, head_dim: int = 128,
                            l2norm_eps: float = 1e-6) -> torch.Tensor:
    """Varlen causal depthwise conv of x (tokens, dim), dim = parts x part_dim.

    weight is (dim, 4) fp32 or (parts, 4, part_dim) (the kda_decode page's
    [qkv, width, channel] copy), any strides; cache_indices may be a strided
    1-D view (the page passes its stride to the kernel).

    Returns (dim // part_dim, tokens, part_dim) in x's dtype; conv_states is
    updated in place.  `activation` "silu", "swish" or True selects SiLU;
    None, False, "none" or "identity" none; anything else is a ValueError.  `null_block_id=None` disables padding detection (the
    library gets a value no cache index can hold).  `out` may be given to
    avoid the allocation.  `use_qk_l2norm` normalises each head_dim-channel
    head of planes 0 and 1 (q and k) per token, y / sqrt(sum y^2 + l2norm_eps)."""
    act = activation_code(activation)
    _check_conv_tensors(x, weight, bias, conv_states, out, part_dim, x.size(0) if x.dim() else 0)
    tokens, dim = x.shape
    num_seqs = max(query_start_loc.numel() - 1, 0)
    _check_vector("query_start_loc", query_start_loc, 0, (torch.int32,))
    _check_vector("cache_indices", cache_indices, num_seqs, (torch.int32,), strided=True)
    _check_vector("has_initial_state", has_initial_state, num_seqs, (torch.bool, torch.uint8))
    _check_devices(x=x, weight=weight, bias=bias, conv_states=conv_states,
                   query_start_loc=query_start_loc, cache_indices=cache_indices,
                   has_initial_state=has_initial_state, out=out)
    if out is None:
        out = torch.empty((dim // part_dim, tokens, part_dim), dtype=x.dtype, device=x.device)
    null = -(2 ** 62) if null_block_id is None else int(null_block_id)
    norm = make_l2norm(0b011, head_dim, l2norm_eps) if use_qk_l2norm else None
    kda_packed_conv1d_l2norm(x, x.stride(0), tokens, dim, part_dim, weight, bias, conv_states,
                             cache_indices, has_initial_state, query_start_loc,
                             num_seqs, null, act, out,
                             layout_of(x, weight, conv_states, cache_indices), norm, stream)
    return out
