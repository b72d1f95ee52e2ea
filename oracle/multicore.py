"""The CPU oracle on every host core (test infrastructure, benchmark only).

Channels of the depthwise conv are independent, so a batch splits into
disjoint channel blocks. Each block is a complete call of the unchanged
oracle, ``packed_conv1d_ex``, on a column slice of x. The weight, bias and
conv-state rows of the block are passed as strided views, with the block as
its only output plane. One worker process per core owns one block. Together
the blocks compute the whole batch once per round. Nothing here changes the
oracle's arithmetic. The harness only runs the oracle on all cores at once,
to time it. The outputs are discarded, and each block's state updates stay
inside its own channels.

Workers are separate interpreters started with subprocess (fork + exec), so
a parent that already holds a CUDA context is safe. The arrays travel as
.npy files in a temporary folder, /dev/shm when it exists. Workers map x
read-only and the conv state read-write, so nothing is copied per worker.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile
import time

import numpy as np

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_ARRAYS = ("x_buf", "weight", "bias", "conv_states", "cache_indices", "has_initial_state",
           "query_start_loc")


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # not Linux
        return os.cpu_count() or 1


def channel_blocks(dim: int, parts: int) -> list[tuple[int, int]]:
    """[c0, c1) ranges that tile 0..dim-1 in `parts` near-equal blocks."""
    parts = max(1, min(parts, dim))
    edges = [round(i * dim / parts) for i in range(parts + 1)]
    return [(edges[i], edges[i + 1]) for i in range(parts) if edges[i + 1] > edges[i]]


class OraclePool:
    """One worker per channel block of batch `b` (a workloads.Batch)."""

    def __init__(self, b, procs: int | None = None, timeout_s: float = 600.0):
        self.procs = procs or host_cores()
        self.timeout_s = timeout_s
        arrays = {"x_buf": b.x_buf, "weight": b.weight,
                  "bias": np.zeros(0, np.float32) if b.bias is None else b.bias,
                  "conv_states": b.conv_states, "cache_indices": b.cache_indices,
                  "has_initial_state": b.has_initial_state,
                  "query_start_loc": b.query_start_loc}
        need = 2 * sum(a.nbytes for a in arrays.values()) + (1 << 20)
        base = None  # the system's temporary folder, unless /dev/shm has room
        if os.path.isdir("/dev/shm") and shutil.disk_usage("/dev/shm").free > need:
            base = "/dev/shm"
        self.dir = tempfile.mkdtemp(prefix="kda_oracle_", dir=base)
        for name in _ARRAYS:
            np.save(os.path.join(self.dir, name + ".npy"), np.ascontiguousarray(arrays[name]))
        meta = [b.x_dtype, b.col_offset, b.dim, int(b.bias is not None), b.null_block_id,
                b.activation]
        with open(os.path.join(self.dir, "meta.txt"), "w") as f:
            f.write(" ".join(str(v) for v in meta))
        self.blocks = channel_blocks(b.dim, self.procs)
        env = dict(os.environ)
        env["PYTHONPATH"] = _ROOT + os.pathsep + env.get("PYTHONPATH", "")
        env["OMP_NUM_THREADS"] = "1"
        self.workers = []
        try:
            for c0, c1 in self.blocks:
                self.workers.append(subprocess.Popen(
                    [sys.executable, "-m", "oracle.multicore", self.dir, str(c0), str(c1)],
                    stdin=subprocess.PIPE, stdout=subprocess.PIPE, text=True, env=env, cwd=_ROOT))
            for w in self.workers:
                self._expect(w, "ready")
        except BaseException:
            self.close()
            raise

    def _expect(self, w, word: str) -> str:
        line = w.stdout.readline().strip()
        if not line.startswith(word):
            raise RuntimeError(f"oracle worker said {line!r}, expected {word!r}")
        return line

    def run(self, reps: int = 1) -> float:
        """Every worker runs its block `reps` times; returns the wall seconds
        from the start command to the last worker's finish."""
        t0 = time.perf_counter()
        for w in self.workers:
            w.stdin.write(f"run {reps}\n")
            w.stdin.flush()
        for w in self.workers:
            self._expect(w, "done")
        return time.perf_counter() - t0

    def states(self) -> np.ndarray:
        """A copy of the conv states as the workers left them."""
        return np.load(os.path.join(self.dir, "conv_states.npy")).copy()

    def close(self) -> None:
        for w in self.workers:
            try:
                w.stdin.write("quit\n")
                w.stdin.flush()
            except (BrokenPipeError, OSError, ValueError):
                pass
        for w in self.workers:
            try:
                w.wait(timeout=self.timeout_s)
            except subprocess.TimeoutExpired:
                w.kill()
                w.wait()
        self.workers = []
        shutil.rmtree(self.dir, ignore_errors=True)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def _worker(folder: str, c0: int, c1: int) -> None:
    import oracle

    lib = oracle.load()
    load = lambda name, mode=None: np.load(os.path.join(folder, name + ".npy"), mmap_mode=mode)
    x_buf = load("x_buf", "r")
    states = load("conv_states", "r+")
    weight, bias = load("weight"), load("bias")
    ci, his, qsl = load("cache_indices"), load("has_initial_state"), load("query_start_loc")
    with open(os.path.join(folder, "meta.txt")) as f:
        x_dtype, col_offset, dim, has_bias, null_block_id, activation = f.read().split()
    dtype = {"bf16": oracle.DTYPE_BF16, "f16": oracle.DTYPE_F16, "f32": oracle.DTYPE_F32}[x_dtype]
    blk = c1 - c0
    w_blk = weight[c0:c1]
    b_blk = bias[c0:c1] if int(has_bias) else None
    s_blk = states[:, c0:c1, :]
    print("ready", flush=True)
    for line in sys.stdin:
        cmd = line.split()
        if not cmd or cmd[0] == "quit":
            break
        reps = int(cmd[1])
        for _ in range(reps):
            oracle.packed_conv1d_ex(np.asarray(x_buf), dtype, int(col_offset) + c0, blk, blk,
                                    w_blk, b_blk, s_blk, ci, his, qsl, int(null_block_id),
                                    int(activation), lib=lib)
        print("done", flush=True)


if __name__ == "__main__":
    _worker(sys.argv[1], int(sys.argv[2]), int(sys.argv[3]))
