"""moe_permute_noalloc -- the dispatch stage for callers that cannot allocate
device memory (its scratch is a fixed array inside the library) -- must give
exactly what moe_permute gives with a caller workspace, on two calls in a row
(the second call must not be disturbed by what the first left in the shared
array), and the oracle's permutation; it keeps moe_permute's shape rules, its
empty-batch behaviour and its handling of an out-of-range expert id.
Collected last so a failure here never hides another test's result."""
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


def test_noalloc_permute_matches_the_oracle():
    """The stable counting sort of the dispatch stage, straight against the
    oracle's permutation (counts, exclusive offsets, perm, inv_perm bit-exact)
    and the gathered rows x_perm[p] = x[perm[p] / K]."""
    import sparse_expert_ffn_moe_gb300 as moe
    T, E, K, d = 1000, 64, 6, 192
    idx, x = _inputs(T, E, K, d, 3)
    s = moe.make_shape(T, d, E, K, 64, 0, "bf16")
    got = _outputs(T, E, K, d)
    moe.moe_permute_noalloc(s, idx, x, got["counts"], got["offsets"], got["perm"], got["inv"],
                            got["x_perm"])
    torch.cuda.synchronize()
    counts, offsets, perm, inv = oracle.permute(idx.cpu().numpy(), E)
    assert np.array_equal(got["counts"].cpu().numpy(), counts)
    assert np.array_equal(got["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(got["perm"].cpu().numpy(), perm)
    assert np.array_equal(got["inv"].cpu().numpy(), inv)
    rows = torch.from_numpy(perm // K).long().cuda()
    assert torch.equal(got["x_perm"], x[rows])


def test_noalloc_permute_with_no_tokens():
    """T = 0: nothing to sort; every count and offset is written as zero."""
    import sparse_expert_ffn_moe_gb300 as moe
    E = 16
    s = moe.make_shape(0, 128, E, 2, 64, 0, "bf16")
    c = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    o = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    moe.moe_permute_noalloc(s, None, None, c, o, None, None, None)
    torch.cuda.synchronize()
    assert torch.count_nonzero(c).item() == 0 and torch.count_nonzero(o).item() == 0


def test_noalloc_permute_drops_an_out_of_range_expert_like_moe_permute():
    """One slot names expert E (out of range).  Both entry points drop it --
    offsets[E] = T*K - 1 and inv_perm[f] = -1 -- and agree on every other
    output; moe_permute records MOE_ERR_BOUNDS in its workspace.  A valid call
    right after gives the oracle's permutation again."""
    import sparse_expert_ffn_moe_gb300 as moe
    T, E, K, d = 300, 32, 4, 128
    idx, x = _inputs(T, E, K, d, 5)
    f_bad = 2 * K + 1
    bad = idx.clone()
    bad.view(-1)[f_bad] = E
    s = moe.make_shape(T, d, E, K, 64, 0, "bf16")
    ref = _outputs(T, E, K, d)
    ws = moe.alloc_workspace(s)
    moe.moe_permute(s, bad, x, ref["counts"], ref["offsets"], ref["perm"], ref["inv"],
                    ref["x_perm"], ws)
    got = _outputs(T, E, K, d)
    moe.moe_permute_noalloc(s, bad, x, got["counts"], got["offsets"], got["perm"], got["inv"],
                            got["x_perm"])
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == moe.MOE_ERR_BOUNDS
    n = T * K
    assert got["offsets"][E].item() == n - 1
    assert got["inv"].view(-1)[f_bad].item() == -1
    for k in ("counts", "offsets", "inv"):
        assert torch.equal(got[k], ref[k]), k
    assert torch.equal(got["perm"][:n - 1], ref["perm"][:n - 1])
    assert torch.equal(got["x_perm"][:n - 1], ref["x_perm"][:n - 1])
    # the next call on the shared scratch starts clean
    again = _outputs(T, E, K, d)
    moe.moe_permute_noalloc(s, idx, x, again["counts"], again["offsets"], again["perm"],
                            again["inv"], again["x_perm"])
    torch.cuda.synchronize()
    counts, offsets, perm, inv = oracle.permute(idx.cpu().numpy(), E)
    assert np.array_equal(again["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(again["perm"].cpu().numpy(), perm)
    assert np.array_equal(again["inv"].cpu().numpy(), inv)


def test_noalloc_permute_refuses_shapes_beyond_its_scratch():
    import sparse_expert_ffn_moe_gb300 as moe
    s = moe.make_shape(1 << 20, 64, 256, 8, 64, 0, "bf16")  # 8M slots: 32 MB of row map
    idx = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = torch.zeros(257, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_permute_noalloc(s, idx, None, c, c, None, None, None)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
    # the shape rules are moe_permute's: inter <= 0 is refused as an invalid argument
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_permute_noalloc(moe.make_shape(4, 64, 8, 2, 0, 0, "bf16"), idx, None, c, c,
                                None, None, None)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
