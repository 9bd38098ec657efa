"""Stage 2 on the GPU (moe_permute): counts, offsets, the stable permutation, its
inverse and the row gather must equal the oracle's bit for bit."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import sparse_expert_ffn_moe_gb300 as m
    return m


def _permute(moe, idx_np: np.ndarray, E: int, d: int = 64, dtype: str = "bf16", with_x=True):
    T, K = idx_np.shape
    s = moe.make_shape(T, d, E, K, 64, 0, dtype)
    ws = moe.alloc_workspace(s)
    idx = torch.from_numpy(np.ascontiguousarray(idx_np)).cuda()
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    n = T * K
    perm = torch.full((max(n, 1),), -1, dtype=torch.int32, device="cuda")
    inv = torch.full((max(n, 1),), -1, dtype=torch.int32, device="cuda")
    x = x_perm = None
    if with_x:
        x = mi.normal((T, d), 1.0, dtype, "cuda", 5, "perm_x")
        x_perm = torch.zeros((max(n, 1), d), dtype=x.dtype, device="cuda")
    moe.moe_permute(s, idx, x, counts, offsets, perm, inv, x_perm, ws)
    torch.cuda.synchronize()
    return dict(counts=counts.cpu().numpy(), offsets=offsets.cpu().numpy(),
                perm=perm.cpu().numpy()[:n], inv=inv.cpu().numpy()[:n],
                x=None if x is None else x.cpu(), x_perm=None if x_perm is None else x_perm.cpu()[:n],
                err=moe.moe_get_device_error(ws))


@pytest.mark.parametrize("T,E,K,scale", [(64, 8, 2, 512), (8, 256, 8, 512), (16384, 256, 8, 512),
                                         (1000, 3, 3, 1), (1, 4, 4, 8), (2048, 1, 1, 8),
                                         (333, 64, 5, 2), (4096, 8, 2, 512), (130, 1024, 32, 4)])
def test_permute_is_bit_exact(moe, T, E, K, scale):
    logits = mi.grid_logits(T, E, seed=201, scale=scale).numpy()
    idx, _, _ = oracle.route(None, None, K, logits_in=logits)
    got = _permute(moe, idx, E)
    counts, offsets, perm, inv = oracle.permute(idx, E)
    assert got["err"] == 0
    assert np.array_equal(got["counts"], counts)
    assert np.array_equal(got["offsets"], offsets)
    assert np.array_equal(got["perm"], perm)
    assert np.array_equal(got["inv"], inv)
    assert torch.equal(got["x_perm"], got["x"][torch.from_numpy(perm // K).long()])


def test_one_expert_takes_every_token(moe):
    T, E, K = 3000, 16, 4
    logits = mi.grid_logits(T, E, seed=202).numpy()
    logits[:, 11] = 100.0
    idx, _, _ = oracle.route(None, None, K, logits_in=logits)
    got = _permute(moe, idx, E)
    counts, offsets, perm, inv = oracle.permute(idx, E)
    assert counts[11] == T
    for k, v in (("counts", counts), ("offsets", offsets), ("perm", perm), ("inv", inv)):
        assert np.array_equal(got[k], v), k


def test_zero_tokens(moe):
    got = _permute(moe, np.zeros((0, 2), np.int32), 8, with_x=False)
    assert np.all(got["counts"] == 0) and np.all(got["offsets"] == 0)


def test_out_of_range_expert_id_is_reported_and_dropped(moe):
    idx = np.array([[0, 1], [1, 9], [2, -1], [3, 0]], np.int32)  # E = 4: 9 and -1 are invalid
    got = _permute(moe, idx, 4)
    assert got["err"] == moe.MOE_ERR_BOUNDS
    assert got["counts"].tolist() == [2, 2, 1, 1]
    assert got["offsets"].tolist() == [0, 2, 4, 5, 6]
    assert got["inv"][3] == -1 and got["inv"][5] == -1
    assert got["perm"][:6].tolist() == [0, 7, 1, 2, 4, 6]
