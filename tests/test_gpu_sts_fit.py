"""GPU parity of the STS temperature fit (dspark_sts_fit) against the oracle
("DSpark：半自回归生成与置信度调度的投机解码", section 校准问题：原始置信度不可靠).

The kernel forms survivals and bin indices in binary32, the oracle in
binary64.  A sample whose exact M * a lies within DELTA_PER_MK * M * k of a
bin edge may land in the neighbouring bin on the device; each such sample can
move the ECE by at most 2/N, so the ECE tolerance is
    ECE_ATOL * k + 2 * (near-edge samples) / N
(the first term covers the binary32 survival error, about k * 6e-7 per
sample, and the fixed-point bin totals).  The chosen index must equal the
oracle's argmin, except where the two ECE values lie within their combined
tolerance: such near-ties are counted and must stay rare.  The oracle is
evaluated with the device's earlier temperatures, so a near-tie at one
position does not propagate.
"""
import numpy as np
import pytest
import torch

import oracle
import workload

pytestmark = pytest.mark.gpu

ECE_ATOL = 1e-6            # per position index k
DELTA_PER_MK = 1e-6        # near-edge window, in units of M * k


@pytest.fixture(scope="module")
def vm():
    import verify_markov_head_gb300 as vm
    return vm


def _grid(G, lo=0.25, hi=4.0):
    return workload.sts_grid(G, lo, hi)


def _fit(vm, score, acc_len, grid, M):
    T, idx, ece = vm.dspark_sts_fit(score.cuda(), acc_len.cuda(), grid.cuda(), M=M)
    torch.cuda.synchronize()
    return T.cpu().numpy(), idx.cpu().numpy(), ece.cpu().numpy()


def _tolerance(score, T_dev, grid, M, cols=None):
    """Per (k, g) tolerance from the oracle's own survivals."""
    N, gamma = score.shape
    g_sel = np.arange(grid.numel()) if cols is None else np.asarray(cols)
    tol = np.zeros((gamma, g_sel.size))
    for k in range(1, gamma + 1):
        a = oracle.sts_survival(score, T_dev[:k - 1], k, grid.numpy().astype(np.float64)[g_sel])
        u = a * M
        r = np.rint(u)
        near = (np.abs(u - r) < DELTA_PER_MK * M * k) & (r >= 1) & (r <= M - 1)
        tol[k - 1] = ECE_ATOL * k + 2.0 * near.sum(axis=0) / N
    return tol


def _check(score, acc_len, grid, M, T_dev, idx_dev, ece_dev, max_near_ties=0):
    gridd = grid.numpy().astype(np.float64)
    assert (T_dev == grid.numpy()[idx_dev]).all()
    ref = oracle.sts_fit(score, acc_len, gridd, M=M, T_fixed=T_dev.astype(np.float64))
    tol = _tolerance(score, T_dev, grid, M)
    err = np.abs(ece_dev - ref["ece"])
    assert (err <= tol).all(), f"max ECE error {err.max():.3e}, worst excess {(err - tol).max():.3e}"
    near_ties = 0
    for k in range(score.shape[1]):
        gi, oi = int(idx_dev[k]), int(ref["idx"][k])
        if gi != oi:
            gap = ref["ece"][k, gi] - ref["ece"][k, oi]
            assert gap <= tol[k, gi] + tol[k, oi], f"position {k + 1}: index {gi} vs {oi}, gap {gap:.3e}"
            near_ties += 1
    assert near_ties <= max_near_ties
    return ref


def test_sts_fit_parity_ragged(vm):
    # Ragged sample count (not a multiple of 32), two candidate chunks (128 + 72).
    score, acc_len = workload.sts_validation(20_011, seed=21)
    grid = _grid(200)
    T, idx, ece = _fit(vm, score, acc_len, grid, 15)
    _check(score, acc_len, grid, 15, T, idx, ece, max_near_ties=1)


@pytest.mark.parametrize("N,gamma,G,M", [(1, 1, 1, 1), (31, 3, 33, 64), (777, 5, 1000, 7), (4096, 16, 64, 15)])
def test_sts_fit_shapes(vm, N, gamma, G, M):
    T_true = [0.8 + 0.15 * k for k in range(gamma)]
    score, acc_len = workload.sts_validation(N, gamma=gamma, seed=N + G, T_true=T_true)
    grid = _grid(G, 0.3, 3.5)
    T, idx, ece = _fit(vm, score, acc_len, grid, M)
    _check(score, acc_len, grid, M, T, idx, ece, max_near_ties=1)


def test_sts_fit_ties_pick_lowest_index(vm):
    score, acc_len = workload.sts_validation(3000, seed=5)
    # Equal grid values tie exactly (integer bin totals): the lower index wins.
    grid = torch.tensor([1.6, 1.6, 0.7, 1.6, 2.2], dtype=torch.float32)
    T, idx, ece = _fit(vm, score, acc_len, grid, 15)
    assert (ece[:, 0] == ece[:, 1]).all() and (ece[:, 0] == ece[:, 3]).all()
    assert not np.isin(idx, [1, 3]).any()
    # Scores of 0 make every temperature equal: index 0 at every position.
    T0, idx0, ece0 = _fit(vm, torch.zeros_like(score), acc_len, torch.tensor([3.0, 1.0, 2.0]), 15)
    assert (idx0 == 0).all() and (ece0 == ece0[:, :1]).all()


def test_sts_fit_recovers_temperatures(vm):
    T_true = [0.5, 2.0, 1.0, 3.0, 1.5]
    score, acc_len = workload.sts_validation(400_000, gamma=5, seed=9, T_true=T_true)
    grid = _grid(16)   # 0.25 apart
    T, idx, ece = _fit(vm, score, acc_len, grid, 15)
    np.testing.assert_allclose(T, T_true, atol=0.25)
    own = oracle.sts_fit(score, acc_len, grid.numpy().astype(np.float64), M=15)
    assert list(own["idx"]) == list(idx)


def test_sts_fit_flags_bad_input(vm):
    score, acc_len = workload.sts_validation(500, gamma=3, seed=1)
    grid = _grid(8)
    ws = torch.zeros(vm.dspark_sts_workspace_bytes(3, 8, 15), dtype=torch.uint8, device="cuda")
    vm.dspark_sts_fit(score.cuda(), acc_len.cuda(), grid.cuda(), M=15, ws=ws)
    assert vm.dspark_sync_status(ws) == (0, 0)
    bad = score.clone()
    bad[7, 1] = float("nan")
    vm.dspark_sts_fit(bad.cuda(), acc_len.cuda(), grid.cuda(), M=15, ws=ws)
    st, bits = vm.dspark_sync_status(ws)
    assert st != 0 and bits & (1 << 3)
    neg = grid.clone()
    neg[2] = -1.0
    vm.dspark_sts_fit(score.cuda(), acc_len.cuda(), neg.cuda(), M=15, ws=ws)
    st, bits = vm.dspark_sync_status(ws)
    assert st != 0 and bits & (1 << 3)


def test_sts_fit_full_size_sampled(vm):
    """The benchmark's fit (2^20 blocks, 256 temperatures, 15 bins), checked on
    sampled candidates: every chosen one plus a spread of others."""
    c = workload.STS_FIT
    score, acc_len = workload.sts_validation(c["N"], gamma=c["gamma"], seed=c["seed"])
    grid = _grid(c["G"], c["lo"], c["hi"])
    T, idx, ece = _fit(vm, score, acc_len, grid, c["M"])
    assert (T == grid.numpy()[idx]).all()
    assert (idx == np.argmin(ece, axis=1)).all()
    cols = np.unique(np.concatenate([idx, [0, 37, 101, 180, c["G"] - 1]]))
    ref = oracle.sts_fit(score, acc_len, grid.numpy().astype(np.float64)[cols], M=c["M"],
                         T_fixed=T.astype(np.float64))
    tol = _tolerance(score, T, grid, c["M"], cols)
    err = np.abs(ece[:, cols] - ref["ece"])
    assert (err <= tol).all(), f"max ECE error {err.max():.3e}"
