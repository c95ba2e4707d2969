"""The allocation-free permute entry point against the workspace one and
against the oracle.

moe_permute_static_scratch serves callers that cannot allocate device memory
(a plugin given only its input and output buffers, or a process whose device
memory is all held by another allocator): its per-block counts live in a
fixed device array inside the library instead of a caller workspace.  This
file is collected last so that a run stopping at the first failure has run
every other test already; it also passes on its own in a fresh process.
"""

import numpy as np
import pytest
import torch

import moe_inputs
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _case(seed, T, H, E, K, special):
    rng = np.random.Generator(np.random.PCG64(seed))
    ids = moe_inputs.uniform_distinct_ids(rng, T, K, E + special).to(DEV)
    tok = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).bfloat16().to(DEV)
    return tok, ids


def test_static_scratch_permute_matches_workspace_permute_on_consecutive_calls(lib):
    # Two calls in a row: the second, smaller one reuses the array that the
    # first left full of its own counts.
    for seed, (T, H, E, K, special) in enumerate([(16384, 256, 64, 8, 0), (3000, 136, 40, 6, 3)]):
        tok, ids = _case(seed, T, H, E, K, special)
        ref = lib.moe_permute(tok, ids, E, special)
        st = lib.new_status()
        got = lib.moe_permute_static_scratch(tok, ids, E, special, dev_status=st)
        assert lib.moe_check_status(st) == lib.MOE_OK
        assert torch.equal(got.expert_offsets, ref.expert_offsets)
        assert torch.equal(got.tokens_per_expert, ref.tokens_per_expert)
        assert torch.equal(got.row_map, ref.row_map)
        n = int(ref.expert_offsets[-1].item())
        assert torch.equal(got.sorted_indices[:n], ref.sorted_indices[:n])
        assert torch.equal(got.permuted[:n], ref.permuted[:n])
        # and bit for bit against the oracle's routing and row gather
        si, rm, tpe, off = O.permute_routing(ids.cpu().numpy(), E, special)
        assert n == len(si)
        assert np.array_equal(got.expert_offsets.cpu().numpy(), off)
        assert np.array_equal(got.tokens_per_expert.cpu().numpy(), tpe)
        assert np.array_equal(got.row_map.cpu().numpy(), rm)
        assert np.array_equal(got.sorted_indices[:n].cpu().numpy(), si)
        want = O.permute_rows(tok.float().cpu().numpy().astype(np.float64), si, K)
        assert np.array_equal(got.permuted[:n].float().cpu().numpy().astype(np.float64), want)


def test_static_scratch_permute_rejects_sizes_past_its_array(lib):
    # ceil(T*K / 512) * E = 512 * 1024 int32 > 65536
    ids = torch.zeros((32768, 8), dtype=torch.int32, device=DEV)
    with pytest.raises(lib.MoeError) as e:
        lib.moe_permute_static_scratch(None, ids, 1024, 0)
    assert e.value.status == lib.MOE_ERR_CAPACITY
