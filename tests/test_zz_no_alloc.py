"""kda_validate_metadata_device_noalloc, the metadata check for callers that
cannot allocate device memory (for example an engine that has reserved the
whole GPU for its own pool), against kda_validate_metadata_device, which
takes its scratch with cudaMallocAsync.  Both are called through the C ABI
on the same device metadata, twice in a row, so the second no-alloc call
runs on the scratch the first one left behind.

This file's name puts it last in collection order: a run that stops at the
first failure has run every other test before it."""

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


def _metadata(seed, n, lines, fault):
    """Device query_start_loc / cache_indices with one planted fault."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 40, size=n)
    qsl = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tokens = int(qsl[-1]) + 3
    ci = rng.permutation(lines)[:n].astype(np.int32)
    ci[rng.random(n) < 0.05] = -1
    s = int(rng.integers(1, n))
    if fault == "duplicate":
        ci[s] = ci[s - 1] if ci[s - 1] >= 0 else 0
        ci[s - 1] = max(int(ci[s - 1]), 0)
    elif fault == "range":
        ci[s] = lines
    elif fault == "offsets":
        qsl[s] = qsl[s + 1] + 1
    return (torch.from_numpy(qsl).cuda(), torch.from_numpy(ci).cuda(), tokens)


@pytest.mark.parametrize("fault", ["none", "duplicate", "range", "offsets"])
def test_noalloc_matches_the_allocating_check_twice(kda, fault):
    """Status and offending sequence equal those of the allocating entry
    point, on two calls in a row with different metadata (the second call
    must not see the first call's claims)."""
    lines = 50000
    first = _metadata(71, 3000, lines, fault)
    second = _metadata(72, 2000, lines, "none" if fault != "none" else "duplicate")
    for qsl, ci, tokens in (first, second):
        want = kda.validate_metadata_device(qsl, ci, tokens, lines, -1)
        got = kda.validate_metadata_device(qsl, ci, tokens, lines, -1, noalloc=True)
        assert got == want, (fault, got, want)
    assert kda.validate_metadata_device(first[0], first[1], first[2], lines, -1,
                                        noalloc=True) == \
        kda.validate_metadata_device(first[0], first[1], first[2], lines, -1)


def test_noalloc_rejects_more_lines_than_its_scratch(kda):
    qsl = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    ci = torch.tensor([0], dtype=torch.int32, device="cuda")
    assert kda.validate_metadata_device(qsl, ci, 1, 1 << 18, -1, noalloc=True) == (0, -1)
    st, _ = kda.validate_metadata_device(qsl, ci, 1, (1 << 18) + 1, -1, noalloc=True)
    assert st == kda.KDA_ERR_UNSUPPORTED
    assert b"static scratch" in kda.lib().kda_last_error_string()
