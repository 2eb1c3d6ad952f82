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
    if case == "prefill":
        return mi.make("prefill").topk_ids, 64
    r = np.random.default_rng(9)
    return r.integers(0, 5, size=(3001, 7)).astype(np.int32), 5


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["prefill", "ragged_repeats"])
def test_route_static_matches_route_two_calls(case):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ids_np, E = _ids(case)
    T, K = ids_np.shape
    sh = hmm.make_shape(T, 8, 8, E, K)
    ids = torch.from_numpy(ids_np).to(dev)

    def outs():
        return (torch.full((E,), -7, dtype=torch.int32, device=dev),
                torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
                torch.full((T * K,), -7, dtype=torch.int32, device=dev),
                torch.full((T * K,), -7, dtype=torch.int32, device=dev))

    # the existing entry point, with a caller workspace and a context
    ctx = hmm.Context.for_device(dev)
    fwd, _, _ = hmm.hmm_workspace_size(sh, False)
    ws = torch.empty(fwd, dtype=torch.uint8, device=dev)
    ref = outs()
    hmm.hmm_route(ctx.handle, sh, ids, *ref, ws)
    torch.cuda.synchronize()

    for call in range(2):
        got = outs()
        hmm.hmm_route_static(sh, ids, *got)
        torch.cuda.synchronize()
        for name, g, r in zip(("counts", "offsets", "slot2row", "row2slot"), got, ref):
            assert torch.equal(g, r), f"call {call}: {name} differs from hmm_route"
