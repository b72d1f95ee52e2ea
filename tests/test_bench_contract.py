"""bench.py's output contract, checked on the CPU.

The reference arm (the oracle on the host cores) runs here on the tiny
workload and must print exactly one JSON line with the keys the benchmark
contract names; under a multi-rank launch only rank 0 prints. Our arm has no
CPU path, so without a GPU it must exit non-zero with a message instead of
printing a number.
"""

from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"}


def _bench(*args, env=None, timeout=300):
    full = dict(os.environ)
    full.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, timeout=timeout, cwd=ROOT, env=full)


def test_reference_arm_prints_one_contract_line():
    r = _bench("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert BASE_KEYS <= set(line), BASE_KEYS - set(line)
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 1 and line["steps"] == 2 and line["warmup"] == 1
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["config"]["workload"] == "tiny"
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["sample"]
    assert cpu["value"] == line["value"] and cpu["unit"] == line["unit"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = _bench("--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "1",
               env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_our_arm_fails_loudly_without_a_gpu():
    r = _bench("--workload", "tiny", "--steps", "3", "--warmup", "3", timeout=120)
    assert r.returncode != 0
    assert r.stdout.strip() == ""  # no number printed
    assert "GPU" in r.stderr


@pytest.mark.parametrize("entry,norm,layout", [
    ("packed", False, ("dense", "channel_major")),
    ("packed", False, ("position_major", "tap_major")),
    ("packed", True, ("dense", "channel_major")),
    ("packed", True, ("position_major", "channel_major")),
    ("update", False, ("dense", "channel_major")),
    ("update", False, ("position_major", "tap_major")),
    ("update", True, ("dense", "channel_major")),
])
def test_prepared_step_matches_the_c_signature(entry, norm, layout):
    """The timed step's prepared C call (bench.prepare) passes exactly the
    arguments its C function declares, for every entry point the bench can
    time.  Host tensors stand in for device ones: nothing is called."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    import linear_attention_prefill_varlen_gb300 as pkg

    old = (bench.ENTRY, bench.NORM, dict(bench.LAYOUT_OPTS))
    try:
        bench.ENTRY = entry
        bench.NORM = pkg.make_l2norm(0b011, 64, 1e-6) if norm else None
        bench.LAYOUT_OPTS.update(state_layout=layout[0], weight_layout=layout[1])
        b = workloads.make_batch("prep", 3, [1] * 4 if entry == "update" else [3, 5],
                                 256, 128, 264, 8)
        s = bench.upload(b, torch.device("cpu"))
        fn, args = bench.prepare(pkg, b, s, 0)
        assert len(args) == len(fn.argtypes), (fn.__name__, len(args), len(fn.argtypes))
        want = {("packed", False): "kda_packed_conv1d", ("update", False): "kda_conv1d_update",
                ("packed", True): "kda_packed_conv1d_l2norm",
                ("update", True): "kda_conv1d_update_l2norm"}[(entry, norm)]
        if entry == "packed" and not norm and layout != ("dense", "channel_major"):
            want = "kda_packed_conv1d_ex"
        assert fn.__name__ == want
    finally:
        bench.ENTRY, bench.NORM = old[0], old[1]
        bench.LAYOUT_OPTS.clear()
        bench.LAYOUT_OPTS.update(old[2])


def test_sized_workload_names():
    """prefill<T> / decode<N> build the 16K chunk's and the decode step's
    shapes at other sizes; other names are rejected by the option parser."""
    import bench
    import workloads

    b = workloads.by_name("prefill4096")
    assert (b.tokens, b.num_seqs, b.dim, b.part_dim, b.row_stride) == (4096, 1, 4608, 1536, 6400)
    d = workloads.by_name("decode256")
    assert (d.tokens, d.num_seqs) == (256, 256) and d.conv_states.shape[0] == 512
    assert workloads.by_name("long16k").name == "long16k"
    for bad in ("prefill0", "prefill", "decode-1", "long8k", "prefill12345678"):
        assert not workloads.valid_name(bad)
        with pytest.raises(SystemExit):
            bench.parse_args(["--workload", bad])
    assert bench.parse_args(["--workload", "decode4096"]).workload == "decode4096"
    # the page's figure covers 2K-16K-token prefill chunks
    assert bench.page_range(workloads.by_name("prefill2048"))
    assert bench.page_range(b)
    assert not bench.page_range(workloads.by_name("prefill32768"))
    assert not bench.page_range(d)
