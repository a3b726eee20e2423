"""moe_permute_static_scratch: the permutation for callers that cannot
allocate device memory (hosted inside a framework whose memory manager owns
every allocation, or in loops that cannot afford cudaMalloc's device-wide
synchronisation).  Its scratch is a fixed array inside the library, so the
test checks, through the C ABI, that it returns exactly what moe_permute
(which takes a caller workspace) returns, on two calls in a row sharing that
array, and that a problem too large for the array is refused.

Collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test.
"""

import numpy as np
import pytest
import torch

from routed_expert_ffn_gemm_gb300 import api, build

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _library():
    build.build()
    api._lib()


def _outputs(T, E, k, d):
    return (torch.empty(E, dtype=torch.int32, device=DEV), torch.empty(E + 1, dtype=torch.int32, device=DEV),
            torch.empty(T * k, dtype=torch.int32, device=DEV), torch.empty(T * k, dtype=torch.int32, device=DEV),
            torch.empty((T * k, d), dtype=torch.bfloat16, device=DEV))


@pytest.mark.parametrize("T,E,k", [(4096, 256, 8), (8192, 128, 8), (64, 8, 2)])
def test_static_scratch_permute_matches_workspace_permute(T, E, k):
    d = 128
    p = api.problem(T, d, 128, E, k)
    ws = api.workspace_for(p)
    rng = np.random.default_rng(T + E)
    for call in range(2):  # two calls in a row share the library's array
        idx = torch.from_numpy(np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)).to(DEV)
        x = torch.randn((T, d), device=DEV).to(torch.bfloat16)
        want = _outputs(T, E, k, d)
        got = _outputs(T, E, k, d)
        api.moe_permute(p, idx, x, *want[:4], want[4], ws)
        api.moe_permute_static_scratch(p, idx, x, *got[:4], got[4])
        torch.cuda.synchronize()
        for a, b in zip(want, got):
            assert torch.equal(a, b), f"call {call}: outputs differ"
    assert api.moe_read_device_status() == 0


def test_static_scratch_permute_refuses_problems_beyond_its_array():
    # ceil(T*k/256) * E = 513 * 1024 > 262144 int32
    T, E, k = 16416, 1024, 8
    p = api.problem(T, 128, 128, E, k)
    idx = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    outs = _outputs(T, E, k, 128)
    with pytest.raises(api.MoEError) as e:
        api.moe_permute_static_scratch(p, idx, None, *outs[:4], None)
    assert e.value.status == api.ERR_WORKSPACE
