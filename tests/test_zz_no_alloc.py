"""The allocation-free routing sort, qmoe_align_sort_static_scratch.

It is meant for callers that cannot allocate device memory when they route
tokens (a host framework that owns all allocations, a plugin that may not
allocate after start-up, a latency path where allocation is forbidden), so
it keeps its scratch in a fixed array inside the library.  These tests call
it through the C ABI and require its outputs to be identical to those of
qmoe_align_sort with a caller workspace, on two calls in a row (the second
call sees the first call's leftovers in the shared array).

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""

import numpy as np
import pytest
import torch

from quantized_mixture_experts_moe_gb300 import binding as qb
from quantized_mixture_experts_moe_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

KEYS = ("counts", "offsets", "sorted_pair_ids", "pair_slot")


def _outputs(E, P, dev):
    return dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
                offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                sorted_pair_ids=torch.empty(P, dtype=torch.int32, device=dev),
                pair_slot=torch.empty(P, dtype=torch.int32, device=dev),
                status=torch.zeros(1, dtype=torch.int32, device=dev))


def _with_workspace(d, ids, dev):
    o = _outputs(d.E, d.T * d.k, dev)
    ws = qb.alloc_workspace(qb.workspace_bytes(d), dev)
    qb.qmoe_align_sort(d, ids, o["counts"], o["offsets"], o["sorted_pair_ids"], o["pair_slot"], o["status"], ws)
    return o


def _static(d, ids, dev):
    o = _outputs(d.E, d.T * d.k, dev)
    qb.qmoe_align_sort_static_scratch(d, ids, o["counts"], o["offsets"], o["sorted_pair_ids"], o["pair_slot"],
                                      o["status"])
    return o


def test_static_scratch_matches_workspace_version_two_calls():
    dev = torch.device("cuda", 0)
    rng = np.random.default_rng(2024)
    cases = [
        (gen.routing_uniform(rng, 4096, 512, 10), 512),   # the prefill layer's routing (40 chunks)
        (gen.routing_zipf(rng, 64, 512, 10), 512),        # skewed decode routing, fewer chunks
    ]
    for ids_np, E in cases:
        T, k = ids_np.shape
        d = qb.dims(T, k, 4096, 1024, E)
        ids = torch.from_numpy(ids_np).to(dev)
        ref = _with_workspace(d, ids, dev)
        first = _static(d, ids, dev)
        second = _static(d, ids, dev)
        torch.cuda.synchronize()
        for out in (first, second):
            for key in KEYS:
                assert torch.equal(out[key], ref[key]), key
            assert int(out["status"].item()) == 0


def test_static_scratch_rejects_shapes_beyond_its_array():
    dev = torch.device("cuda", 0)
    # ceil(P / 2048) * E * 4 bytes must fit the array
    E = 4096
    chunks = qb.STATIC_SCRATCH_BYTES // (4 * E) + 1
    T, k = chunks * 2048 // 8, 8
    d = qb.dims(T, k, 4096, 1024, E)
    ids = torch.zeros((T, k), dtype=torch.int32, device=dev)
    o = _outputs(E, T * k, dev)
    with pytest.raises(qb.QmoeError, match="-2"):
        qb.qmoe_align_sort_static_scratch(d, ids, o["counts"], o["offsets"], o["sorted_pair_ids"], o["pair_slot"],
                                          o["status"])
