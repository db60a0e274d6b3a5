"""moe_permute_noalloc: the permute for callers that cannot allocate device memory
(engine plugins that own every allocation, code running during CUDA-graph capture,
fixed-budget serving paths).  Its index scratch is a static device array inside the
library instead of a caller workspace.  Checked through the C ABI against moe_permute on
two calls in a row with different shapes (the shared array keeps the previous call's
contents, which must not matter), plus the rejection of a shape too large for it.
Collected last on purpose: it runs alone or after every other test."""
import numpy as np
import pytest
import torch

import combine_moe_route_softmax_gb300 as moe
from gpu_helpers import need_gpu

pytestmark = pytest.mark.gpu


def noalloc_permute(idx, E, x, with_shared, out_dtype):
    """Call moe_permute_noalloc through the C ABI; outputs allocated here by the caller."""
    T, K = idx.shape
    H = x.shape[1]
    cap = T * K + (T if with_shared else 0)
    fp8 = out_dtype == moe.MOE_E4M3
    out = dict(
        xp=torch.zeros(cap, H, dtype=torch.uint8 if fp8 else torch.bfloat16, device="cuda"),
        xp_scales=torch.zeros(cap, H // 128, dtype=torch.float32, device="cuda") if fp8 else None,
        cu_seqlens=torch.empty(E + int(with_shared) + 1, dtype=torch.int32, device="cuda"),
        src_row=torch.empty(cap, dtype=torch.int32, device="cuda"),
        inv_map=torch.empty(T, K, dtype=torch.int32, device="cuda"),
        shared_map=torch.empty(T, dtype=torch.int32, device="cuda") if with_shared else None)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = lambda t: None if t is None else t.data_ptr()
    rc = moe.lib().moe_permute_noalloc(p(idx), T, K, E, int(with_shared), p(x), H, out_dtype, p(out["xp"]),
                                       p(out["xp_scales"]), p(out["cu_seqlens"]), p(out["src_row"]),
                                       p(out["inv_map"]), p(out["shared_map"]), p(status),
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == 0, moe.STATUS.get(rc, rc)
    return out, status


def problem(T, K, E, seed, pad):
    g = torch.Generator().manual_seed(seed)
    idx = torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)]).to(torch.int32)
    idx[torch.rand(T, K, generator=g) < pad] = -1
    x = torch.randn(T, 512, generator=g).to(torch.bfloat16)
    return idx.cuda(), x.cuda()


@pytest.mark.parametrize("out_dtype", [moe.MOE_BF16, moe.MOE_E4M3])
def test_noalloc_permute_matches_workspace_permute(out_dtype):
    need_gpu()
    # two calls in a row: a large shape, then a small one that reuses the same static array
    for (T, K, E, shared, pad, seed) in [(16384, 8, 256, True, 0.5, 1), (300, 6, 40, False, 0.1, 2)]:
        idx, x = problem(T, K, E, seed, pad)
        st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
        want = moe.moe_permute(idx, E, x, with_shared=shared, out_dtype=out_dtype, dev_status=st_ref)
        got, st = noalloc_permute(idx, E, x, shared, out_dtype)
        torch.cuda.synchronize()
        assert st.item() == st_ref.item() == 0
        N = int(want["cu_seqlens"][-1].item())
        for key in ("cu_seqlens", "src_row", "inv_map", "shared_map"):
            if want[key] is not None:
                assert torch.equal(got[key], want[key]), key
        # permute is bit-exact: the rows it wrote must be identical
        assert torch.equal(got["xp"][:N].view(torch.uint8), want["xp"][:N].view(torch.uint8))
        if out_dtype == moe.MOE_E4M3:
            assert torch.equal(got["xp_scales"][:N], want["xp_scales"][:N])


def test_noalloc_rejects_shapes_beyond_its_scratch():
    need_gpu()
    L = moe.lib()
    limit = L.moe_permute_noalloc_max_scratch_bytes()
    assert limit == 1 << 20
    T, K, E = 65536, 8, 1024                       # needs 4 MiB of index scratch
    assert L.moe_permute_workspace_bytes(T, K, E, 1) > limit
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    rc = L.moe_permute_noalloc(dummy.data_ptr(), T, K, E, 1, dummy.data_ptr(), 512, moe.MOE_BF16,
                               dummy.data_ptr(), None, dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
                               dummy.data_ptr(), None, torch.cuda.current_stream().cuda_stream)
    assert rc == 2                                 # MOE_ERR_WORKSPACE, nothing launched
    assert np.all(dummy.cpu().numpy() == 0)
