"""kda_validate_metadata_device (device metadata, checks on the GPU) against
kda_validate_metadata (host metadata, the same checks in plain C) on valid and
malformed metadata: the same status and the same offending sequence."""

from __future__ import annotations

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_attention_prefill_varlen_gb300 as pkg

    pkg.lib()
    return pkg


def _both(kda, qsl, ci, tokens, lines, null=-1, stride=1):
    host = kda.validate_metadata(torch.tensor(qsl, dtype=torch.int32),
                                 torch.tensor(ci, dtype=torch.int32), tokens, lines, null)
    ci_np = np.asarray(ci, dtype=np.int32)
    buf = torch.full((max(len(ci_np) * stride, 1),), 7, dtype=torch.int32, device="cuda")
    view = buf[::stride][:len(ci_np)]
    view.copy_(torch.from_numpy(ci_np))
    dev = kda.validate_metadata_device(torch.tensor(qsl, dtype=torch.int32, device="cuda"), view,
                                       tokens, lines, null)
    return host, dev


CASES = [
    ([0, 2, 5], [0, 1], 8, 4),          # valid
    ([0, 6, 5], [0, 1], 8, 4),          # offsets go backwards at 1
    ([-1, 2, 5], [0, 1], 8, 4),         # negative first offset
    ([0, 2, 9], [0, 1], 8, 4),          # last offset beyond tokens
    ([0, 2, 5], [0, 4], 8, 4),          # line out of range
    ([0, 2, 5], [-2, 1], 8, 4),         # negative line (not the null block)
    ([0, 2, 5], [1, 1], 8, 4),          # duplicate line
    ([0, 2, 5], [-1, -1], 8, 4),        # two null blocks are not a duplicate
    ([0, 1, 1, 3, 3], [3, -1, 0, 2], 3, 4),
    ([0, 3, 2, 9], [5, 5, 9], 8, 4),    # offsets fail first: reported before the lines
]


@pytest.mark.parametrize("stride", [1, 3])
@pytest.mark.parametrize("case", CASES)
def test_device_check_matches_host_check(kda, case, stride):
    qsl, ci, tokens, lines = case
    host, dev = _both(kda, qsl, ci, tokens, lines, stride=stride)
    assert host == dev, (case, host, dev)


def test_device_check_random_batches(kda):
    """Seeded random metadata, each with one planted fault of a random kind
    (or none), over up to 5000 sequences and 20000 lines."""
    rng = np.random.default_rng(23)
    for trial in range(60):
        n = int(rng.integers(1, 5000))
        lines = int(rng.integers(n, 4 * n + 10))
        lens = rng.integers(0, 50, size=n)
        qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        tokens = int(qsl[-1] + rng.integers(0, 5))
        ci = rng.permutation(lines)[:n].astype(np.int64)
        ci[rng.random(n) < 0.05] = -1
        kind = trial % 5
        s = int(rng.integers(0, n))
        if kind == 1:
            ci[s] = ci[(s + 1) % n] if n > 1 else lines  # duplicate (or out of range)
        elif kind == 2:
            ci[s] = lines + int(rng.integers(0, 3))
        elif kind == 3 and n > 1:
            qsl[s + 1] = qsl[s] - 1
        elif kind == 4:
            tokens = int(qsl[-1]) - 1
        host, dev = _both(kda, qsl.tolist(), ci.tolist(), tokens, lines,
                          stride=1 + trial % 2)
        assert host == dev, (trial, kind, host, dev)


def test_device_check_empty_and_bad_arguments(kda):
    e = torch.zeros(0, dtype=torch.int32, device="cuda")
    assert kda.validate_metadata_device(torch.zeros(1, dtype=torch.int32, device="cuda"), e, 0,
                                        4, -1) == (0, -1)
    st, _ = kda.validate_metadata_device(torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                                         torch.tensor([0], dtype=torch.int32, device="cuda"),
                                         1, -5, -1)
    assert st == kda.KDA_ERR_INVALID_ARG
