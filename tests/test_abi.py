"""The C-ABI library loads on the CPU, exports every function that
include/moe_route.h declares, and rejects bad arguments on the host (before
any CUDA call, so no GPU is needed)."""
import os
import re
import subprocess

import pytest

from padded_permute_combine_gb300 import _lib
from padded_permute_combine_gb300 import build as libbuild


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return _lib.load()


def test_header_and_exports_agree(lib):
    declared = _lib.header_functions()
    assert len(declared) == len(set(declared)) == 22
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = [f for f in declared if f not in exported]
    assert not missing, missing
    assert set(declared) == set(_lib.SIGNATURES)
    for f in declared:
        assert getattr(lib, f) is not None


def test_informational_calls(lib):
    assert lib.moe_version() == 100
    assert lib.moe_error_string(0) == b"ok"
    assert lib.moe_error_string(1) == b"invalid argument"
    assert lib.moe_error_string(99) == b"unknown error"
    assert lib.moe_route_build_workspace_size(65536, 256) > 0
    assert lib.moe_route_build_workspace_size(-1, 256) == 0
    assert lib.moe_route_build_workspace_size(10, 0) == 0
    assert lib.moe_route_build_workspace_size(10, _lib.MOE_MAX_EXPERTS + 1) == 0
    assert lib.moe_scatter_workspace_size(65536) >= 65536 * 4
    assert lib.moe_route_build_gather_workspace_size(65536, 256) >= lib.moe_route_build_workspace_size(65536, 256)
    assert lib.moe_route_build_gather_workspace_size(-1, 256) == 0


FAKE = 1 << 20  # an aligned non-null address; never dereferenced (host checks fail first)


def test_host_validation_rejects_bad_arguments(lib):
    ws = lib.moe_route_build_workspace_size(8, 4)
    # negative n, E out of range, pad multiple 0, missing outputs, small workspace, misaligned pointer
    assert lib.moe_route_build(FAKE, -1, 4, 1, FAKE, FAKE, FAKE, None, None, FAKE, ws, None, None) == 1
    assert lib.moe_route_build(FAKE, 8, 0, 1, FAKE, FAKE, FAKE, None, None, FAKE, ws, None, None) == 1
    assert lib.moe_route_build(FAKE, 8, 5000, 1, FAKE, FAKE, FAKE, None, None, FAKE, ws, None, None) == 1
    assert lib.moe_route_build(FAKE, 8, 4, 0, FAKE, FAKE, FAKE, None, None, FAKE, ws, None, None) == 1
    assert lib.moe_route_build(FAKE, 8, 4, 1, None, FAKE, FAKE, None, None, FAKE, ws, None, None) == 1
    assert lib.moe_route_build(FAKE, 8, 4, 1, FAKE, FAKE, FAKE, None, None, FAKE, 0, None, None) == 1
    assert lib.moe_route_build(FAKE + 2, 8, 4, 1, FAKE, FAKE, FAKE, None, None, FAKE, ws, None, None) == 2
    assert lib.moe_route_build(FAKE, 2**31, 4, 1, FAKE, FAKE, FAKE, None, None, FAKE, 1 << 40, None, None) == 1
    # padded total overflowing int32
    assert lib.moe_route_build(FAKE, 2**31 - 10, 4, 8, FAKE, FAKE, FAKE, FAKE, None, FAKE, 1 << 40, None, None) == 1
    # gather: bad dtype, negative capacity, top_k out of range, T*K overflow, misaligned x
    assert lib.moe_binned_gather(FAKE, 7, FAKE, FAKE, None, 4, 8, 2, 2, 1, FAKE, None, None) == 2
    assert lib.moe_binned_gather(FAKE, 0, FAKE, FAKE, None, 4, 8, 2, -1, 1, FAKE, None, None) == 1
    assert lib.moe_binned_gather(FAKE, 0, FAKE, FAKE, None, 4, 8, 2, 2, 0, FAKE, None, None) == 1
    assert lib.moe_binned_gather(FAKE, 0, FAKE, FAKE, None, 4, 8, 2, 2, 65, FAKE, None, None) == 1
    assert lib.moe_binned_gather(FAKE, 0, FAKE, FAKE, None, 2**30, 8, 2, 2, 4, FAKE, None, None) == 1
    assert lib.moe_binned_gather(FAKE + 2, 0, FAKE, FAKE, None, 4, 8, 2, 2, 1, FAKE, None, None) == 2
    assert lib.moe_padded_gather(FAKE, 1, FAKE, FAKE, None, None, 4, 8, 2, 1, FAKE, 8, None, None) == 1
    assert lib.moe_padded_gather(FAKE, 1, FAKE, FAKE, FAKE, None, 4, 8, 2, 1, FAKE, -1, None, None) == 1
    # misaligned positions
    assert lib.moe_binned_gather(FAKE, 0, FAKE, FAKE, FAKE + 2, 4, 8, 2, 2, 1, FAKE, None, None) == 2
    assert lib.moe_padded_gather(FAKE, 0, FAKE, FAKE, FAKE, FAKE + 2, 4, 8, 2, 1, FAKE, 8, None, None) == 2
    assert lib.moe_padded_wgrad(FAKE, FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE + 2, 4, 8, 2, 1, 8, FAKE, None,
                                None) == 2
    # scatter without positions needs a workspace
    assert lib.moe_binned_scatter(FAKE, 0, FAKE, FAKE, FAKE, None, None, 4, 8, 2, 4, 1, FAKE, None, 0, None,
                                  None) == 1
    assert lib.moe_padded_scatter(FAKE, 1, FAKE, FAKE, FAKE, None, None, None, 4, 8, 2, 1, 8, FAKE, None, 0, None,
                                  None) == 1
    assert lib.moe_binned_wgrad(FAKE, None, 0, FAKE, FAKE, FAKE, 4, 8, 2, 4, 1, FAKE, None, None) == 1
    assert lib.moe_padded_wgrad(FAKE, FAKE, 0, FAKE, FAKE, FAKE, FAKE, None, 4, 8, 2, 1, -3, FAKE, None, None) == 1
    # weighted gather: weights required when there are tokens; misaligned weights
    assert lib.moe_binned_gather_weighted(FAKE, 1, FAKE, FAKE, None, None, 4, 8, 2, 2, 1, FAKE, None, None) == 1
    assert lib.moe_binned_gather_weighted(FAKE, 1, FAKE, FAKE, FAKE + 2, None, 4, 8, 2, 2, 1, FAKE, None, None) == 2
    assert lib.moe_padded_gather_weighted(FAKE, 0, FAKE, FAKE, None, FAKE, None, 4, 8, 2, 1, FAKE, 8, None, None) == 1
    assert lib.moe_padded_gather_weighted(FAKE, 0, FAKE, FAKE, FAKE, None, None, 4, 8, 2, 1, FAKE, 8, None, None) == 1
    # route build + gather in one call: positions required, padded_bins required for the padded layout,
    # bad dtype, workspace too small, negative out_rows (all before anything is enqueued)
    ws2 = lib.moe_route_build_workspace_size(8, 2)
    assert lib.moe_route_build_binned_gather(FAKE, FAKE, 0, 4, 8, 2, 2, 2, 1, FAKE, FAKE, FAKE, None, None, FAKE,
                                             FAKE, ws2, None, None) == 1
    assert lib.moe_route_build_binned_gather(FAKE, FAKE, 9, 4, 8, 2, 2, 2, 1, FAKE, FAKE, FAKE, None, FAKE, FAKE,
                                             FAKE, ws2, None, None) == 2
    assert lib.moe_route_build_binned_gather(FAKE, FAKE, 0, 4, 8, 2, 2, 2, 1, FAKE, FAKE, FAKE, None, FAKE, FAKE,
                                             FAKE, 0, None, None) == 1
    assert lib.moe_route_build_binned_gather(FAKE, FAKE, 0, 4, 8, 2, 2, -1, 1, FAKE, FAKE, FAKE, None, FAKE, FAKE,
                                             FAKE, ws2, None, None) == 1
    assert lib.moe_route_build_padded_gather(FAKE, FAKE, 1, 4, 8, 2, 2, 4, FAKE, FAKE, FAKE, None, FAKE, FAKE, 16,
                                             FAKE, ws2, None, None) == 1
    assert lib.moe_route_build_padded_gather(FAKE, FAKE, 1, 4, 8, 2, 2, 4, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, -1,
                                             FAKE, ws2, None, None) == 1
    # routing check: status word required, E out of range, negative n, misaligned bins
    assert lib.moe_check_routing(FAKE, FAKE, FAKE, None, None, 8, 2, None, None) == 1
    assert lib.moe_check_routing(FAKE, FAKE, FAKE, None, None, 8, 0, FAKE, None) == 1
    assert lib.moe_check_routing(FAKE, FAKE, FAKE, None, None, -1, 2, FAKE, None) == 1
    assert lib.moe_check_routing(FAKE, FAKE, FAKE + 2, None, None, 8, 2, FAKE, None) == 2
    # gating: top_k above E, bad mode, E above the gating limit
    assert lib.moe_topk_gating(FAKE, 4, 8, 9, 0, 1, FAKE, FAKE, None) == 1
    assert lib.moe_topk_gating(FAKE, 4, 8, 2, 5, 1, FAKE, FAKE, None) == 1
    assert lib.moe_topk_gating(FAKE, 4, 2048, 2, 0, 1, FAKE, FAKE, None) == 2
    assert lib.moe_topk_gating(FAKE, 0, 8, 2, 1, 0, FAKE, FAKE, None) == 0
    assert lib.moe_routing_map_to_indices_fwd(FAKE, FAKE, -1, 4, 2, FAKE, FAKE, None) == 1
    assert lib.moe_routing_map_to_indices_fwd(FAKE, FAKE, 4, 4, 0, FAKE, FAKE, None) == 1
    assert lib.moe_routing_map_to_indices_fwd(FAKE + 1, FAKE, 4, 4, 2, FAKE, FAKE, None) == 2
    assert lib.moe_routing_map_to_indices_bwd(FAKE, FAKE, 4, 0, 2, FAKE, None, None) == 1
    assert lib.moe_routing_map_to_indices_bwd(FAKE, None, 4, 4, 2, FAKE, None, None) == 1


def test_empty_problems_enqueue_nothing(lib):
    # Zero rows / zero tokens return MOE_OK without launching anything.
    assert lib.moe_binned_gather(FAKE, 0, FAKE, FAKE, None, 4, 8, 2, 0, 1, FAKE, None, None) == 0
    assert lib.moe_padded_gather(FAKE, 0, FAKE, FAKE, FAKE, None, 4, 8, 2, 1, FAKE, 0, None, None) == 0
    assert lib.moe_binned_scatter(FAKE, 0, FAKE, FAKE, FAKE, None, FAKE, 0, 8, 2, 4, 1, FAKE, None, 0, None,
                                  None) == 0
    assert lib.moe_binned_wgrad(FAKE, FAKE, 0, FAKE, FAKE, FAKE, 0, 8, 2, 4, 1, FAKE, None, None) == 0
    assert lib.moe_routing_map_to_indices_fwd(FAKE, FAKE, 0, 4, 2, FAKE, FAKE, None) == 0
    assert lib.moe_routing_map_to_indices_bwd(FAKE, FAKE, 0, 4, 2, FAKE, None, None) == 0


def test_product_path_has_no_oracle_dependency():
    import glob
    import os

    pkg = os.path.dirname(_lib.__file__)
    for f in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if f.endswith((".py", ".cu", ".cuh", ".h")):
            txt = open(f).read()
            assert not re.search(r"^\s*(import|from)\s+oracle\b", txt, flags=re.M), f
            assert "liboracle" not in txt and "oracle.c" not in txt, f


def test_loader_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load(str(tmp_path / "missing.so"))


def test_header_is_plain_c(tmp_path):
    """include/moe_route.h compiles as C11 in a plain C host (no C++, no
    torch): the C host under tests/c_abi builds with gcc -c."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    subprocess.run([gcc, "-std=c11", "-Wall", "-Werror", "-c", "-I", os.path.join(root, "include"), "-I",
                    os.path.join(cuda, "include"), os.path.join(here, "c_abi", "route_and_gather.c"), "-o",
                    str(tmp_path / "host.o")], check=True)
