"""GPU parity of block_table_update (dirty-tracked table synchronisation).

FlexiCache blog summary (MLSys'26), "System design, head-level block table":
only the changed entries of the [batch, layer, head, logical_block] table are
synchronised.  The kernel must leave exactly the oracle's table, with the
changed entries in device memory or read from pinned host memory, and skip
and report invalid updates.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_minmax_gb300 import kvmm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    from paged_kv_cache_minmax_gb300 import build

    build.build_library()
    kvmm.load()
    oracle.build()
    yield


@pytest.mark.parametrize("where,frac", [("device", 0.02), ("pinned", 0.02), ("pinned", 0.5), ("device", 0.0)])
def test_changed_entries_reach_the_device_table(where, frac):
    B, L, Hkv, Pmax, n_phys = 3, 4, 8, 300, 20000
    shape = kvmm.make_shape(B, L, 2 * Hkv, Hkv, 128, 16, Pmax, 64, n_phys)
    rng = np.random.default_rng(int(frac * 100) + len(where))
    old = rng.integers(-1, n_phys, size=(B, L, Hkv, Pmax)).astype(np.int32)
    new = old.copy()
    pick = rng.random(new.shape) < frac
    new[pick] = rng.integers(-1, n_phys, size=int(pick.sum()))
    idx = np.flatnonzero(old != new).astype(np.int64)
    rng.shuffle(idx)
    val = new.ravel()[idx].astype(np.int32)
    table = torch.tensor(old, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ti, tv = torch.tensor(idx), torch.tensor(val)
    if where == "device":
        ti, tv = ti.cuda(), tv.cuda()
    else:
        ti, tv = ti.pin_memory(), tv.pin_memory()
    kvmm.block_table_update(shape, ti, tv, table, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = old.copy()
    assert oracle.table_update(want, n_phys, idx, val) == 0
    np.testing.assert_array_equal(table.cpu().numpy(), want)
    np.testing.assert_array_equal(want, new)


def test_invalid_updates_are_skipped_and_reported():
    B, L, Hkv, Pmax, n_phys = 1, 1, 2, 16, 50
    shape = kvmm.make_shape(B, L, 2, Hkv, 64, 16, Pmax, 8, n_phys)
    table = torch.zeros(B, L, Hkv, Pmax, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.tensor([3, B * L * Hkv * Pmax, 5, -1], dtype=torch.int64, device="cuda")
    val = torch.tensor([7, 1, n_phys, 2], dtype=torch.int32, device="cuda")
    kvmm.block_table_update(shape, idx, val, table, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvmm.ERR_OUT_OF_RANGE
    t = table.view(-1).cpu().numpy()
    assert t[3] == 7 and t[5] == 0 and (np.delete(t, 3) == 0).all()
