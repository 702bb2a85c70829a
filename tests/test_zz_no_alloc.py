"""The workspace-free permute (moe_permute_no_alloc), for callers that cannot
allocate device memory, must give exactly what moe_permute gives.

Called through the C ABI with ctypes, twice in a row on different inputs (the
internal scratch keeps the previous call's contents, which must not matter).
This file is collected last so a failure here stops a -x run only after every
other test has run; it also passes on its own in a fresh process."""
import ctypes as C

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    import moe_routed_expert_gb300 as M
    return M.load()


def _p(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def run_both(lib, T, H, k, E, seed, with_x=True):
    import torch
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[rng.random(ids.shape) < 0.1] = -1
    dev = "cuda"
    tids = torch.from_numpy(ids).to(dev)
    x = torch.randn(T, H, device=dev).to(torch.bfloat16) if with_x else None
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)

    def outs():
        return (torch.full((T * k, H), -3.0, dtype=torch.bfloat16, device=dev) if with_x else None,
                torch.full((E,), -7, dtype=torch.int64, device=dev),
                torch.full((T * k,), -9, dtype=torch.int32, device=dev),
                torch.full((T * k,), -9, dtype=torch.int32, device=dev))

    ref, got = outs(), outs()
    ws_bytes = lib.moe_permute_workspace_size(T, k, E)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    assert lib.moe_permute(_p(x), _p(tids), T, H, k, E, _p(ref[0]), _p(ref[1]), _p(ref[2]), _p(ref[3]),
                           _p(ws), ws_bytes, stream) == 0
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    assert lib.moe_permute_no_alloc(_p(x), _p(tids), T, H, k, E, _p(got[0]), _p(got[1]), _p(got[2]), _p(got[3]),
                                    _p(status), stream) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    R = int(ref[1].sum().item())
    for a, b in zip(ref[1:], got[1:]):
        assert torch.equal(a, b)
    if with_x:
        assert torch.equal(ref[0][:R], got[0][:R])
    return R


def test_no_alloc_permute_matches_moe_permute_on_two_calls(lib):
    # a large call, then a smaller one whose counters sit where the first left data
    R1 = run_both(lib, T=16384, H=512, k=8, E=64, seed=1)
    R2 = run_both(lib, T=300, H=264, k=4, E=37, seed=2)
    assert R1 > 0 and R2 > 0
    run_both(lib, T=999, H=0, k=2, E=8, seed=3, with_x=False)


def test_no_alloc_permute_rejects_sizes_beyond_its_scratch(lib):
    import torch
    # ceil(T*k/1024) * E above 131072 counters: refused on the host, nothing launched
    fake = C.c_void_p(0x10000)
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.moe_permute_no_alloc(None, fake, 1 << 20, 0, 8, 1024, None, fake, fake, fake, None, stream) == 3
    assert lib.moe_permute_no_alloc(None, None, 16, 0, 2, 8, None, fake, fake, fake, None, stream) == 1


def test_no_alloc_permute_bad_id_null_status_empty_batch_and_binding(lib):
    import torch
    import moe_routed_expert_gb300 as M
    dev = "cuda"
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    T, H, k, E = 40, 64, 2, 8
    ids = torch.from_numpy(np.stack([np.arange(k) + (t % (E - k)) for t in range(T)]).astype(np.int32)).to(dev)
    x = torch.randn(T, H, device=dev).to(torch.bfloat16)
    # an id equal to E: the device status word records MOE_ERR_DEVICE
    bad = ids.clone()
    bad[3, 1] = E
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    M.moe_permute_no_alloc(x, bad, E, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 5
    # no status word at all: the same call runs and the good ids are ranked as moe_permute ranks them
    got = M.moe_permute_no_alloc(x, ids, E, device_status=None)
    want = M.moe_permute(x, ids, E)
    torch.cuda.synchronize()
    R = int(want[1].sum().item())
    assert R == T * k
    for a, b in zip(want[1:], got[1:]):
        assert torch.equal(a, b)
    assert torch.equal(want[0][:R], got[0][:R])
    # an empty batch: every expert gets zero rows, and the row tensors may be NULL
    gl = torch.full((E,), -7, dtype=torch.int64, device=dev)
    assert lib.moe_permute_no_alloc(None, None, 0, H, k, E, None, _p(gl), None, None, None, stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(gl, torch.zeros(E, dtype=torch.int64, device=dev))
    # a status word that is not 4-byte aligned is refused on the host
    odd = C.c_void_p(status.data_ptr() + 2)
    assert lib.moe_permute_no_alloc(None, _p(ids), T, 0, k, E, None, _p(gl), _p(got[2]), _p(got[3]), odd,
                                    stream) == 2
