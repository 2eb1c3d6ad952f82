"""The C-ABI library: builds for sm_103a, loads without a GPU, exports every
entry point include/hmm.h declares, and its host-side checks (no device work)
reject bad shapes with the documented codes."""
import os
import re
import shutil

import pytest

import dispatch_grouped_gemm_gb300 as hmm
from dispatch_grouped_gemm_gb300 import build as hbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hmm.h")


def _declared():
    with open(HEADER) as f:
        src = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(hmm_\w+)\s*\(", src, re.M)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        if not os.path.exists(hbuild.LIB):
            pytest.skip("nvcc not available and libhmm.so not built")
    else:
        hbuild.build()
    return hmm.load_library()


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("hmm_create", "hmm_destroy", "hmm_set_option", "hmm_workspace_size", "hmm_route",
              "hmm_forward", "hmm_backward", "hmm_status", "hmm_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), f"libhmm.so does not export {n}"


def test_library_has_no_torch_dependency(lib):
    # the C ABI is plain pointers and sizes: the shared library links no torch
    with open(hbuild.LIB, "rb") as f:
        blob = f.read()
    assert b"libtorch" not in blob and b"libc10" not in blob


def _ws(T=64, H=128, I=64, E=8, K=2, wd=0, training=True):
    return hmm.hmm_workspace_size(hmm.make_shape(T, H, I, E, K, wd), training)


def test_workspace_sizes_consistent(lib):
    f, s, b = _ws()
    assert f > 0 and s > 0 and b > 0
    f0, s0, b0 = _ws(training=False)
    assert s0 == 0 and b0 == 0 and f0 > f          # inference keeps activations in the workspace
    f2, s2, _ = _ws(T=128)
    assert s2 > s and f2 > f
    assert _ws(T=0)[0] >= 0


@pytest.mark.parametrize("kw,code", [
    (dict(H=100), -4), (dict(I=60), -4),            # not multiples of 8 -> layout
    (dict(E=0), -2), (dict(K=0), -2), (dict(T=-1), -2), (dict(E=2000), -2), (dict(K=33), -2),
    (dict(wd=7), -3),
])
def test_workspace_size_rejects_bad_shapes(lib, kw, code):
    with pytest.raises(hmm.HmmError) as ei:
        _ws(**kw)
    assert ei.value.code == code


def test_error_strings(lib):
    for c in range(0, -10, -1):
        assert hmm.hmm_error_string(c)
    assert "unknown" in hmm.hmm_error_string(-99)


def test_phase_names(lib):
    """Phase ids name the launch phases in step order; bench.py keys its
    per-kernel roofline on these names."""
    names = [hmm.hmm_phase_name(i) for i in range(hmm._C["HMM_NUM_PHASES"])]
    assert names == ["route", "dispatch_x", "gemm_fwd", "combine_y", "dispatch_dy",
                     "gemm_bwd_data", "gemm_bwd_weight", "combine_dx"]
    assert hmm.hmm_phase_name(-1) is None
    assert hmm.hmm_phase_name(len(names)) is None


def test_create_without_gpu_fails_cleanly(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(hmm.HmmError) as ei:
        hmm.hmm_create(0)
    assert ei.value.code == -9
