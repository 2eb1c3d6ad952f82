"""hmm_route_static: the routing step for callers that cannot allocate device
memory, such as an engine whose memory pool owns the whole GPU or a plug-in
whose host gives it no allocator.  It keeps its scratch in one fixed array
inside the library instead of a caller workspace, so every call reuses the
contents the previous call left there.  These tests check that it returns
exactly what hmm_route returns (integer outputs, so bit for bit) on two calls
in a row, and that a shape too large for the array is refused up front.

This file sorts last so that a run stopping at its first failure has already
run every other test."""
import numpy as np
import pytest
import torch

import dispatch_grouped_gemm_gb300 as hmm
import moe_inputs as mi


def test_route_static_refuses_shapes_beyond_its_scratch():
    # 2M tokens x 8 slots needs far more than the 8 MiB array; the check
    # happens on the host before any device work (the pointers are never used)
    sh = hmm.make_shape(1 << 21, 8, 8, 64, 8)
    with pytest.raises(hmm.HmmError) as ei:
        hmm.hmm_route_static(sh, 16, 16, 16, 16, 16, stream=0)
    assert ei.value.code == -5


def _ids(case):
    r = np.random.default_rng(9)
    if case == "prefill":
        return mi.make("prefill").topk_ids, 64
    if case == "ragged_repeats":
        return r.integers(0, 5, size=(3001, 7)).astype(np.int32), 5
    # the routing paths with a separate scan launch between the count and
    # rank kernels: more than 512 experts, and more than 32768 chunk x
    # expert histogram entries
    if case == "scan_launch_wide_E":
        return r.integers(0, 600, size=(3000, 6)).astype(np.int32), 600
    if case == "scan_launch_many_chunks":
        return r.integers(0, 256, size=(20000, 8)).astype(np.int32), 256
    if case == "no_tokens":
        return np.zeros((0, 4), np.int32), 16
    raise ValueError(case)


def _outs(E, S, dev):
    return (torch.full((E,), -7, dtype=torch.int32, device=dev),
            torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
            torch.full((max(S, 1),), -7, dtype=torch.int32, device=dev),
            torch.full((max(S, 1),), -7, dtype=torch.int32, device=dev))


def _route(sh, ids, E, S, dev):
    """The existing entry point, with a caller workspace and a context."""
    ctx = hmm.Context.for_device(dev)
    fwd, _, _ = hmm.hmm_workspace_size(sh, False)
    ws = torch.empty(max(fwd, 256), dtype=torch.uint8, device=dev)
    ref = _outs(E, S, dev)
    hmm.hmm_route(ctx.handle, sh, ids, *ref, ws)
    torch.cuda.synchronize()
    return ref


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["prefill", "ragged_repeats", "scan_launch_wide_E",
                                  "scan_launch_many_chunks", "no_tokens"])
def test_route_static_matches_route_two_calls(case):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ids_np, E = _ids(case)
    T, K = ids_np.shape
    S = T * K
    sh = hmm.make_shape(T, 8, 8, E, K)
    ids = torch.from_numpy(ids_np).to(dev)
    ref = _route(sh, ids, E, S, dev)

    # a first call on a larger shape with other ids leaves its contents in the
    # shared array, so the calls below start from stale scratch
    r = np.random.default_rng(31)
    big_np = r.integers(0, 200, size=(9000, 8)).astype(np.int32)
    big = torch.from_numpy(big_np).to(dev)
    hmm.hmm_route_static(hmm.make_shape(9000, 8, 8, 200, 8), big, *_outs(200, 9000 * 8, dev))
    torch.cuda.synchronize()

    got = [_outs(E, S, dev) for _ in range(2)]
    free0, _ = torch.cuda.mem_get_info(dev)
    for call in range(2):
        hmm.hmm_route_static(sh, ids, *got[call])
        torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0, "device memory changed across hmm_route_static calls"
    for call in range(2):
        for name, g, rr in zip(("counts", "offsets", "slot2row", "row2slot"), got[call], ref):
            assert torch.equal(g, rr), f"call {call}: {name} differs from hmm_route"
