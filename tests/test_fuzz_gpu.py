"""Seeded random configurations, every option of the C ABI at once, against
the oracle.

Each case draws sizes (dim a multiple of 64 up to 1024, part_dim a divisor
that is a multiple of 64), sequence lengths with zeros, short and long
ones, x's type, the conv state's type, width and memory order, the weight's
memory order, bias or none, SiLU or none, a null block, the L2 norm (plane
mask and head size) or none, and the entry point (packed or decode update).
The bar is the one the other parity tests use: states bit-exact, outputs
bit-exact without activation or norm, else within one ulp of bf16 / fp16 or
2^-19 relative for fp32.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import pins
import workloads
from gpu_helpers import assert_states_equal, state_to_device, state_to_host, ulp_diff

pytestmark = pytest.mark.gpu

N_CASES = 120
DT = {"bf16": 0, "f16": 1, "f32": 2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_attention_prefill_varlen_gb300 as pkg

    pkg.lib()


def _draw(i: int) -> dict:
    rng = np.random.default_rng(9000 + i)
    part_dim = int(rng.choice([64, 128, 192, 256]))
    dim = part_dim * int(rng.integers(1, 5))
    while dim > 1024:
        dim -= part_dim
    entry = "update" if rng.random() < 0.3 else "packed"
    if entry == "update":
        lengths = [1] * int(rng.integers(1, 60))
    else:
        n = int(rng.integers(1, 12))
        kinds = rng.choice(["zero", "short", "mid", "long"], size=n, p=[0.1, 0.4, 0.3, 0.2])
        lengths = [0 if k == "zero" else int(rng.integers(1, 6)) if k == "short"
                   else int(rng.integers(6, 80)) if k == "mid" else int(rng.integers(80, 400))
                   for k in kinds]
    heads = [h for h in (16, 32, 64, 128) if part_dim % h == 0]
    norm = None
    if rng.random() < 0.35:
        planes = dim // part_dim
        mask = int(rng.integers(1, 1 << planes))
        norm = (mask, int(rng.choice(heads)), float(np.float32(rng.choice([1e-6, 1e-3, 0.5]))))
    x_dtype = str(rng.choice(["bf16", "f16", "f32"], p=[0.5, 0.25, 0.25]))
    quantum = 4 if x_dtype == "f32" else 8
    return dict(
        seed=9100 + i, lengths=lengths, dim=dim, part_dim=part_dim, entry=entry,
        row_stride=dim + quantum * int(rng.integers(0, 4)),
        col_offset=quantum * int(rng.integers(0, 3)),
        x_dtype=x_dtype,
        state_dtype=str(rng.choice(["f32", "bf16"], p=[0.6, 0.4])),
        state_width=int(rng.choice([3, 3, 4, 5, 8])),
        state_order=str(rng.choice(["dense", "position_major"])),
        weight_order=str(rng.choice(["channel_major", "tap_major"])),
        bias=bool(rng.random() < 0.7), activation=int(rng.random() < 0.7),
        null_count=int(rng.random() < 0.5), his_p=float(rng.choice([0.0, 0.5, 1.0])),
        norm=norm)


def _batch(cfg: dict) -> workloads.Batch:
    n = len(cfg["lengths"])
    b = workloads.make_batch(
        f"fuzz{cfg['seed']}", cfg["seed"], cfg["lengths"], cfg["dim"], cfg["part_dim"],
        cfg["row_stride"] + cfg["col_offset"], 2 * n + 3, col_offset=cfg["col_offset"],
        bias_std=0.1 if cfg["bias"] else None, activation=cfg["activation"],
        his_p=1.0 if cfg["entry"] == "update" else cfg["his_p"],
        null_count=min(cfg["null_count"], n), x_dtype=cfg["x_dtype"],
        state_width=cfg["state_width"], state_dtype=cfg["state_dtype"])
    if cfg["entry"] == "update":
        b.has_initial_state[:] = 1
    return b


def _run_device(b: workloads.Batch, cfg: dict):
    import linear_attention_prefill_varlen_gb300 as pkg

    dev = torch.device("cuda")
    f32 = b.x_dtype == "f32"
    x = torch.from_numpy(b.x_buf if f32 else b.x_buf.view(np.int16)).to(dev)
    out = torch.full((b.dim // b.part_dim, b.tokens, b.part_dim), float("nan") if f32 else -1,
                     dtype=torch.float32 if f32 else torch.int16, device=dev)
    if cfg["state_order"] == "position_major":
        st = state_to_device(np.ascontiguousarray(b.conv_states.transpose(0, 2, 1)), dev)
        st = st.transpose(1, 2)
    else:
        st = state_to_device(b.conv_states, dev)
    if cfg["weight_order"] == "tap_major":
        w = torch.from_numpy(np.ascontiguousarray(b.weight.T)).to(dev).t()
    else:
        w = torch.from_numpy(b.weight).to(dev)
    bias = None if b.bias is None else torch.from_numpy(b.bias).to(dev)
    layout = pkg.make_layout(DT[b.x_dtype], st.size(2), st.stride(), w.stride(),
                             pkg.KDA_DTYPE_BF16 if st.dtype == torch.bfloat16 else
                             pkg.KDA_DTYPE_F32)
    norm = None if cfg["norm"] is None else pkg.make_l2norm(*cfg["norm"])
    xp = x.data_ptr() + (4 if f32 else 2) * b.col_offset
    ci = torch.from_numpy(b.cache_indices).to(dev)
    if cfg["entry"] == "update":
        pkg.kda_conv1d_update_l2norm(xp, b.row_stride, b.tokens, b.dim, b.part_dim, w, bias, st,
                                     ci, b.null_block_id, b.activation, out, layout, norm)
    else:
        his = torch.from_numpy(b.has_initial_state).to(dev)
        qsl = torch.from_numpy(b.query_start_loc).to(dev)
        pkg.kda_packed_conv1d_l2norm(xp, b.row_stride, b.tokens, b.dim, b.part_dim, w, bias, st,
                                     ci, his, qsl, b.num_seqs, b.null_block_id, b.activation,
                                     out, layout, norm)
    torch.cuda.synchronize()
    return out.cpu().numpy(), state_to_host(st)


def _compare(b: workloads.Batch, got: np.ndarray, want: np.ndarray, mask: int) -> None:
    for plane in range(b.dim // b.part_dim):
        normed = bool((mask >> plane) & 1)
        exact = not normed and b.activation == 0
        g, w = got[plane], want[plane]
        if b.x_dtype == "f32":
            unwritten = np.isnan(w)
            assert np.isnan(g[unwritten]).all(), "rows outside sequences written"
            g, w = g[~unwritten], w[~unwritten]
            if exact:
                assert np.array_equal(g.view(np.uint32), w.view(np.uint32)), plane
            else:
                rel = np.abs(g.astype(np.float64) - w) / np.maximum(np.abs(w.astype(np.float64)),
                                                                   1e-30)
                assert (rel <= 2.0 ** -19).all(), (plane, float(rel.max()))
        else:
            gb = g.view(np.uint16)
            untouched = w == 0xFFFF
            assert np.array_equal(gb[untouched], w[untouched]), "rows outside sequences written"
            d = ulp_diff(gb, w)
            assert d.max() <= (0 if exact else 1), (plane, int(d.max()))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_configuration(i):
    cfg = _draw(i)
    b = _batch(cfg)
    st = b.conv_states.copy()
    if cfg["norm"] is None:
        want = pins.run_oracle_ex(b, states=st)["out"]
        mask = 0
    else:
        want = pins.run_oracle_l2norm(b, *cfg["norm"], states=st)["out"]
        mask = cfg["norm"][0]
    got, got_st = _run_device(b, cfg)
    assert_states_equal(got_st, st)
    _compare(b, got, want, mask)
