"""moe_permute_static_scratch: the grouping step for callers that cannot
allocate device memory (for example a server that reserved the GPU's memory
for its own pool, or a plugin host that passes a kernel only its inputs and
outputs).  Its scratch table lives in a fixed array inside the library.

Called through the C ABI and compared with moe_permute (which takes its
scratch from a caller-provided workspace) on two calls in a row, which share
the fixed array.  The grouping is integer work, so the comparison is exact.
This file is collected last so that a failure here cannot hide others."""

import ctypes

import pytest
import torch

from mixture_experts_layer_20_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from mixture_experts_layer_20_gb300 import binding
    return binding


def _call_c_abi(moe, ids, E, x, status, d=None):
    """Direct ctypes call of the exported symbol (no binding helper).  x may be
    None (no gather; d then gives the row width the call is told)."""
    T, k = ids.shape
    d = x.shape[1] if x is not None else d
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * k, dtype=torch.int32, device="cuda")
    slot_pos = torch.empty((T, k), dtype=torch.int32, device="cuda")
    x_perm = torch.empty((T * k, d), dtype=torch.bfloat16, device="cuda") if x is not None else None
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    st = moe._lib.moe_permute_static_scratch(
        p(ids), p(x), T, d, E, k, p(counts), p(offsets), p(perm), p(slot_pos), p(x_perm),
        p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, (counts, offsets, perm, slot_pos, x_perm)


@pytest.mark.parametrize("T,E,k,d", [(6000, 128, 8, 256), (333, 256, 8, 128)])
def test_static_scratch_matches_workspace_version(moe, T, E, k, d):
    for call in range(2):       # two calls in a row share the library's array
        ids, _ = W.random_routing(T, E, k, seed=100 * call + T)
        ids[: T // 4] = ids[0]  # skewed: some experts hot, some empty
        ids = ids.cuda()
        x = W.make_x(W.Workload("n", T, d, E, k, 64, seed=call), device="cuda")
        want = moe.moe_permute(ids, E, x=x)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        st, got = _call_c_abi(moe, ids, E, x, status)
        assert st == moe.MOE_OK, moe._lib.moe_last_error()
        torch.cuda.synchronize()
        for a, b in zip(got, want):
            assert torch.equal(a, b)
        assert status.item() == 0


def test_static_scratch_at_the_table_limit(moe):
    """E = 256 and T*k = 262,144: ceil(T*k/1024) * E = 65,536 entries, the
    whole fixed table.  Two calls in a row, bit for bit against moe_permute."""
    T, k, E = 32768, 8, 256
    for call in range(2):
        ids, _ = W.random_routing(T, E, k, seed=31 + call)
        ids[: T // 8] = ids[1]  # one group of experts hot
        ids = ids.cuda()
        want = moe.moe_permute(ids, E)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        st, got = _call_c_abi(moe, ids, E, None, status, d=64)
        assert st == moe.MOE_OK, moe._lib.moe_last_error()
        torch.cuda.synchronize()
        for a, b in zip(got[:4], want[:4]):
            assert torch.equal(a, b)
        assert status.item() == 0


def test_static_scratch_flags_out_of_range_ids(moe):
    """Several chunks (T*k = 5600 > 4096 takes the two-kernel path) with two
    expert ids out of range: the caller's status word gets bit 2 (device
    check) and the call returns without a fault."""
    T, k, E = 700, 8, 32
    ids, _ = W.random_routing(T, E, k, seed=5)
    ids[5, 3] = E + 3
    ids[600, 0] = -1
    ids = ids.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    st, _ = _call_c_abi(moe, ids, E, None, status, d=64)
    assert st == moe.MOE_OK, moe._lib.moe_last_error()
    torch.cuda.synchronize()
    assert status.item() & 2


def test_static_scratch_without_status_word(moe):
    ids, _ = W.random_routing(100, 16, 4, seed=9)
    ids = ids.cuda()
    want = moe.moe_permute(ids, 16)
    got = moe.moe_permute_static_scratch(ids, 16)
    torch.cuda.synchronize()
    for a, b in zip(got[:4], want[:4]):
        assert torch.equal(a, b)


def test_static_scratch_rejects_sizes_beyond_its_table(moe):
    # ceil(T*k/1024) * E = 257 * 256 > 65536 table entries; nothing is launched
    T, k, E = 1024 * 257 // 8, 8, 256
    ids = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    st = moe._lib.moe_permute_static_scratch(
        ctypes.c_void_p(ids.data_ptr()), None, T, 64, E, k, ctypes.c_void_p(ids.data_ptr()),
        ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(ids.data_ptr()),
        ctypes.c_void_p(ids.data_ptr()), None, None, None)
    assert st == moe.MOE_ERR_UNSUPPORTED
    assert b"exceeds" in moe._lib.moe_last_error()
