"""moe_permute_static_scratch: the permutation for callers that cannot
allocate device memory (hosted inside a framework whose memory manager owns
every allocation, or in loops that cannot afford cudaMalloc's device-wide
synchronisation).  Its scratch is a fixed array inside the library, so the
test checks, through the C ABI, that it returns exactly what the CPU
reference's permutation maps give and what moe_permute (which takes a
caller workspace) returns, on two calls in a row sharing that array; that a
problem filling the array exactly is accepted; and that one chunk more is
refused.

Collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.
"""

import numpy as np
import pytest
import torch

import oracle
from routed_expert_ffn_gemm_gb300 import api, build

pytestmark = pytest.mark.gpu
DEV = "cuda"

# int32 entries of the library's built-in array, and the rows per chunk of
# the large-batch permutation (ceil(T*k / 256) * E entries are needed)
ARRAY_INTS = 262144
CHUNK_ROWS = 256


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()
    api._lib()


def _outputs(T, E, k, d):
    return (torch.empty(E, dtype=torch.int32, device=DEV), torch.empty(E + 1, dtype=torch.int32, device=DEV),
            torch.empty(T * k, dtype=torch.int32, device=DEV), torch.empty(T * k, dtype=torch.int32, device=DEV),
            torch.empty((T * k, d), dtype=torch.bfloat16, device=DEV))


# (8192, 1024, 8): 256 chunks of 256 rows x 1024 experts fill the array exactly
@pytest.mark.parametrize("T,E,k", [(4096, 256, 8), (8192, 128, 8), (64, 8, 2), (8192, 1024, 8)])
def test_static_scratch_permute_matches_oracle_and_workspace_permute(T, E, k):
    d = 128
    p = api.problem(T, d, 128, E, k)
    ws = api.workspace_for(p)
    rng = np.random.default_rng(T + E)
    for call in range(2):  # two calls in a row share the library's array
        idx_np = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        idx = torch.from_numpy(idx_np).to(DEV)
        x = torch.randn((T, d), device=DEV).to(torch.bfloat16)
        want = _outputs(T, E, k, d)
        got = _outputs(T, E, k, d)
        api.moe_permute(p, idx, x, *want[:4], want[4], ws)
        api.moe_permute_static_scratch(p, idx, x, *got[:4], got[4])
        torch.cuda.synchronize()
        # bit-exact against the CPU reference's maps (stable counting sort)
        counts_r, offsets_r, perm_r, inv_r = oracle.permutation_maps(idx_np, E)
        assert np.array_equal(got[0].cpu().numpy(), counts_r), f"call {call}: counts"
        assert np.array_equal(got[1].cpu().numpy(), offsets_r), f"call {call}: offsets"
        assert np.array_equal(got[2].cpu().numpy(), perm_r), f"call {call}: perm_token"
        assert np.array_equal(got[3].cpu().numpy().reshape(T, k), inv_r), f"call {call}: inv_row"
        assert torch.equal(got[4].cpu(), x.cpu()[torch.from_numpy(perm_r.astype(np.int64))]), f"call {call}: rows"
        # and the same bits as the workspace entry point
        for a, b in zip(want, got):
            assert torch.equal(a, b), f"call {call}: outputs differ"
    assert api.moe_read_device_status() == 0


@pytest.mark.parametrize("T,E,k", [
    (8193, 1024, 8),    # 257 chunks x 1024 experts: one chunk past the array
    (16416, 1024, 8),   # 513 chunks x 1024 experts: twice the array
])
def test_static_scratch_permute_refuses_problems_beyond_its_array(T, E, k):
    assert -(-T * k // CHUNK_ROWS) * E > ARRAY_INTS
    p = api.problem(T, 128, 128, E, k)
    idx = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    outs = _outputs(T, E, k, 128)
    with pytest.raises(api.MoEError) as e:
        api.moe_permute_static_scratch(p, idx, None, *outs[:4], None)
    assert e.value.status == api.ERR_WORKSPACE


def test_static_scratch_permute_checks_the_problem_like_moe_permute():
    # a problem moe_permute refuses (ffn not a multiple of 8) is refused the
    # same way, before the scratch-size check
    p = api.problem(64, 128, 100, 8, 2)
    outs = _outputs(64, 8, 2, 128)
    idx = torch.zeros((64, 2), dtype=torch.int32, device=DEV)
    with pytest.raises(api.MoEError) as a:
        api.moe_permute(p, idx, None, *outs[:4], None, None)
    with pytest.raises(api.MoEError) as b:
        api.moe_permute_static_scratch(p, idx, None, *outs[:4], None)
    assert a.value.status == b.value.status == api.ERR_UNSUPPORTED
