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


# Non-null stand-ins for device pointers: the calls below return before any
# CUDA call, so nothing is ever dereferenced.  P is 16-byte aligned, U is not.
P, U = 0x10000, 0x10008
F32, BF16 = 0, 1
INV, SHAPE, UNSUP, CAP = 1, 2, 3, 4
HOST_CHECKS = [
    # (entry point, arguments, status) -- the rule each case breaks
    ("moe_selftest_bounded_wait", (None, None), INV),                       # no status word
    ("moe_gate_up_swiglu", (P, BF16, P, 128, 128, 64, 1025, P, P, P, None, None, None), SHAPE),  # E > 1024
    ("moe_gate_up_swiglu", (P, BF16, P, 128, 128, 64, 2, P, P, U, None, None, None), INV),       # act unaligned
    ("moe_gate_up_swiglu", (P, F32, P, 16, 6, 64, 2, P, P, P, None, None, None), SHAPE),         # fp32 H % 4
    ("moe_down_proj", (P, BF16, None, 128, 128, 64, 2, P, P, None, None), INV),                  # no offsets
    ("moe_down_dgrad_swiglu", (P, P, F32, P, 128, 64, 64, 2, P, P, None, None), UNSUP),          # bf16 only
    ("moe_gate_up_dgrad", (P, F32, P, 128, 64, 64, 2, P, P, P, None, None), UNSUP),              # bf16 only
    ("moe_down_wgrad", (P, P, BF16, P, 128, 64, 64, 2, None, None, None), INV),                  # no dW_down
    ("moe_gate_up_wgrad", (P, P, BF16, P, 128, 64, 64, 2, U, P, None, None), INV),               # dW_gate unaligned
    ("moe_shared_expert_mlp", (P, 16, 96, 64, P, P, P, P, P, None, None), SHAPE),                # H % 64
    ("moe_shared_expert_mlp", (P, -1, 128, 64, P, P, P, P, P, None, None), INV),                 # T < 0
    ("moe_gate_up_swiglu_gather", (P, 16, P, 0, P, 128, 128, 64, 2, P, P, P, None, None, None), INV),  # K = 0
    ("moe_gate_up_swiglu_gather", (U, 16, P, 2, P, 128, 128, 64, 2, P, P, P, None, None, None), INV),  # tokens unaligned
    ("moe_gate_up_wgrad_gather", (P, P, 16, None, 2, P, 128, 128, 64, 2, P, P, None, None), INV),      # no indices
    ("moe_unpermute_grad", (P, P, BF16, P, P, 4, 64, 17, 68, P, P, None), SHAPE),                # K > 16
    ("moe_unpermute", (P, BF16, P, P, 4, 4, 2, 8, P, None), SHAPE),                              # 8-byte rows
    ("moe_combine", (P, BF16, P, P, P, None, None, 4, 64, 2, 8, 0, 0, 0, 0, None, None, None, P, None, None), INV),  # E = 0
    ("moe_combine", (P, BF16, P, P, P, None, None, 4, 64, 2, 8, 8, 0, 2, 0, None, None, None, P, None, None), INV),  # copy experts, no ori_x
    ("moe_combine", (P, BF16, P, P, P, None, None, 4, 64, 4, 8, 2, 0, 0, 0, None, None, None, P, None, None), SHAPE),  # K > E + specials
    ("moe_combine_masked", (P, BF16, P, P, P, None, None, P, 3, 4, 64, 2, 8, 8, 0, 0, 0, None, None, None, P, None, None), INV),  # mask_dims 3
    ("moe_permute_masked", (P, BF16, P, 4, 64, 2, 8, 0, P, 0, P, P, P, P, P, P, 1 << 20, None, None), INV),  # mask_dims 0
    ("moe_permute", (P, BF16, P, 4, 64, 2, 8, 0, P, P, P, P, P, P, 0, None, None), INV),         # workspace too small
    ("moe_permute", (P, BF16, P, 4, 64, 2, 8, 0, P, P, P, P, P, U, 1 << 20, None, None), INV),   # workspace unaligned
    ("moe_permute", (P, BF16, P, 4, 64, 4, 2, 1, P, P, P, P, P, P, 1 << 20, None, None), SHAPE),  # K > E + specials
    ("moe_permute_static_scratch", (P, BF16, P, 1 << 20, 64, 8, 1024, 0, P, P, P, P, P, None, None), CAP),  # scratch too small
    ("moe_invert_sorted_indices", (P, 10, 8, P, None), INV),                                     # N > T*K
    ("moe_permute_indices_window", (P, 2, 8, 6, 4, P, 16, P, P, None, None), SHAPE),             # window past E_all
    ("moe_permute_indices", (P, 0, 8, P, 16, P, P, None, None), INV),                           # R = 0
]


@pytest.mark.parametrize("name,args,status", HOST_CHECKS,
                         ids=[f"{c[0]}-{i}" for i, c in enumerate(HOST_CHECKS)])
def test_entry_points_reject_bad_arguments_on_the_host(built_lib, name, args, status):
    """Each entry point's documented argument rules, broken one at a time,
    return their status before any CUDA call (so this runs without a GPU)."""
    from unpermute_moe_permute_gb300 import binding
    lib = binding.load_library(built_lib)
    assert getattr(lib, name)(*args) == status


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
