"""moe_permute_noalloc -- the dispatch stage for callers that cannot allocate
device memory (its scratch is a fixed array inside the library) -- must give
exactly what moe_permute gives with a caller workspace, on two calls in a row
(the second call must not be disturbed by what the first left in the shared
array).  Collected last so a failure here never hides another test's result."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle

pytestmark = pytest.mark.gpu


def _inputs(T, E, K, d, seed):
    logits = mi.grid_logits(T, E, seed=seed, scale=4).numpy()
    idx, _, _ = oracle.route(None, None, K, logits_in=logits)
    x = mi.normal((T, d), 1.0, "bf16", "cuda", seed, "noalloc_x")
    return torch.from_numpy(idx).cuda(), x


def _outputs(T, E, K, d):
    n = T * K
    z = lambda *s: torch.full(s, -1, dtype=torch.int32, device="cuda")  # noqa: E731
    return dict(counts=z(E), offsets=z(E + 1), perm=z(n), inv=z(n),
                x_perm=torch.zeros((n, d), dtype=torch.bfloat16, device="cuda"))


@pytest.mark.parametrize("pass_inv", [True, False])
def test_noalloc_permute_matches_workspace_permute_twice(pass_inv):
    import sparse_expert_ffn_moe_gb300 as moe
    for (T, E, K, d, seed) in ((4096, 256, 8, 256, 1), (333, 8, 2, 128, 2)):
        idx, x = _inputs(T, E, K, d, seed)
        s = moe.make_shape(T, d, E, K, 64, 0, "bf16")
        ref = _outputs(T, E, K, d)
        ws = moe.alloc_workspace(s)
        moe.moe_permute(s, idx, x, ref["counts"], ref["offsets"], ref["perm"], ref["inv"],
                        ref["x_perm"], ws)
        got = _outputs(T, E, K, d)
        moe.moe_permute_noalloc(s, idx, x, got["counts"], got["offsets"], got["perm"],
                                got["inv"] if pass_inv else None, got["x_perm"])
        torch.cuda.synchronize()
        for k in ("counts", "offsets", "perm", "x_perm") + (("inv",) if pass_inv else ()):
            assert torch.equal(got[k], ref[k]), (T, k)


def test_noalloc_permute_refuses_shapes_beyond_its_scratch():
    import sparse_expert_ffn_moe_gb300 as moe
    s = moe.make_shape(1 << 20, 64, 256, 8, 64, 0, "bf16")  # 8M slots: 32 MB of row map
    idx = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = torch.zeros(257, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_permute_noalloc(s, idx, None, c, c, None, None, None)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
