"""The C-ABI library builds, loads without a GPU and exports every function
the public header declares; the oracle and the CUDA path share no code."""

import ast
import glob
import os
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built_lib():
    from unpermute_moe_permute_gb300 import build
    if not os.path.exists(build.LIB_PATH):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("library not built and nvcc not available")
        build.build()
    return build.LIB_PATH


def test_header_declares_the_hot_path_calls():
    from unpermute_moe_permute_gb300.binding import header_symbols
    names = set(header_symbols())
    for required in ["moe_permute", "moe_expert_mlp", "moe_gate_up_swiglu", "moe_down_proj",
                     "moe_unpermute", "moe_unpermute_grad", "moe_combine",
                     "moe_permute_indices", "moe_permute_grad", "moe_expert_mlp_grad",
                     "moe_check_status"]:
        assert required in names


def test_library_exports_every_header_symbol(built_lib):
    from unpermute_moe_permute_gb300 import binding
    lib = binding.load_library(built_lib)
    for name in binding.header_symbols():
        assert hasattr(lib, name), f"{name} declared in the header but not exported"
        assert name in binding._SIGNATURES, f"{name} has no ctypes signature in the binding"
    assert lib.moe_abi_version() >= 1
    assert lib.moe_status_string(binding.MOE_ERR_BAD_ID) == b"expert id out of range or repeated in a row"
    # 512-slot blocks: int32 expert counts per block, then one 8-byte flag per block
    assert lib.moe_permute_workspace_size(16384, 8, 64) == 256 * 64 * 4 + 256 * 8


def test_host_side_argument_checks_need_no_gpu(built_lib):
    """Arguments rejected on the host return a status before any CUDA call."""
    from unpermute_moe_permute_gb300 import binding
    lib = binding.load_library(built_lib)
    # K = 17 > 16
    rc = lib.moe_permute(None, 1, None, 4, 64, 17, 64, 0, None, None, None, None, None, None, 0,
                         None, None)
    assert rc == binding.MOE_ERR_SHAPE
    # bad dtype for unpermute
    assert lib.moe_unpermute(None, 9, None, None, 4, 64, 2, 8, None, None) == binding.MOE_ERR_INVALID_ARG
    # bf16 GEMMs need H % 64 == 0 (a dummy, never dereferenced offsets pointer)
    assert lib.moe_gate_up_swiglu(None, 1, 256, 0, 72, 64, 4, None, None, None, None, None,
                                  None) == binding.MOE_ERR_SHAPE
    # R*E above the index kernel's limit
    assert lib.moe_permute_indices(None, 64, 64, None, 0, None, None, None, None) == binding.MOE_ERR_SHAPE


def _imports(path):
    tree = ast.parse(open(path).read())
    mods = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            mods.update(a.name for a in node.names)
        elif isinstance(node, ast.ImportFrom):
            mods.add(("." * node.level) + (node.module or ""))
    return mods


def test_oracle_and_cuda_path_are_independent():
    for f in glob.glob(os.path.join(ROOT, "oracle", "*.py")):
        for m in _imports(f):
            assert "unpermute_moe_permute_gb300" not in m, f
            assert "moe_inputs" not in m, f
    for f in glob.glob(os.path.join(ROOT, "unpermute_moe_permute_gb300", "*.py")):
        for m in _imports(f):
            assert not m.startswith("oracle"), f
    for f in glob.glob(os.path.join(ROOT, "unpermute_moe_permute_gb300", "csrc", "*")):
        assert "oracle" not in open(f).read().lower(), f
