"""Shared helpers for the parity tests: move seeded inputs to the device,
bring results back, and compare with the oracle under the pages' tolerance."""
import numpy as np

import oracle as O

# Tolerance of the pages' own fused-vs-eager bf16 test ("NPU Training Operators
# - GMM", sections "结论" and "验证项"): rtol = atol = 1e-2, applied elementwise as
# |gpu - oracle| <= atol + rtol * |oracle|.
RTOL = 1e-2
ATOL = 1e-2


def dev_bf16(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host_f64(t):
    """bf16 / fp32 / int device tensor -> numpy (bf16 and fp32 as float64)."""
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return O.bf16_bits_to_f64(t.view(torch.int16).numpy().view(np.uint16))
    if t.dtype == torch.float32:
        return t.numpy().astype(np.float64)
    return t.numpy()


def f64(bits):
    return O.bf16_bits_to_f64(bits)


def assert_close(name, got, want, rtol=RTOL, atol=ATOL):
    got = host_f64(got) if not isinstance(got, np.ndarray) else got
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite values" % name
    excess = np.abs(got - want) - (atol + rtol * np.abs(want))
    if np.any(excess > 0):
        i = np.unravel_index(np.argmax(excess), excess.shape)
        n = int(np.sum(excess > 0))
        raise AssertionError("%s: %d of %d elements outside tolerance; worst at %s: got %r want %r"
                             % (name, n, excess.size, i, float(got[i]), float(want[i])))


# ----------------------------------------------------------------------------
# Guard regions (a stand-in for a memory checker): every device tensor the
# binding allocates (outputs and workspaces) is carved out of a larger buffer
# whose bytes before and after it hold a canary pattern; after the test the
# pattern must be intact, so no kernel wrote outside the tensors it was given.
GUARD_BYTES = 4096
CANARY = 0xA5


class GuardedAlloc:
    def __init__(self):
        self.regions = []

    def make(self, shape, dtype, device, fill=None):
        import math
        import torch
        shape = tuple(int(s) for s in shape)
        nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        buf = torch.full((nbytes + 2 * GUARD_BYTES,), CANARY, dtype=torch.uint8, device=device)
        t = buf[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(shape)
        if fill is not None:
            t.fill_(fill)
        self.regions.append((buf, nbytes))
        return t

    def check(self):
        import torch
        torch.cuda.synchronize()
        for i, (buf, nbytes) in enumerate(self.regions):
            head, tail = buf[:GUARD_BYTES], buf[GUARD_BYTES + nbytes:]
            bad_head = int((head != CANARY).sum())
            bad_tail = int((tail != CANARY).sum())
            assert bad_head == 0 and bad_tail == 0, (
                "allocation %d (%d bytes): %d guard bytes before it and %d after it were overwritten"
                % (i, nbytes, bad_head, bad_tail))


class GuardedTorch:
    """torch, with empty / empty_like / zeros on a CUDA device returning
    guarded tensors (everything else passes through)."""

    def __init__(self, torch_mod, alloc):
        self._t = torch_mod
        self._a = alloc

    def __getattr__(self, name):
        return getattr(self._t, name)

    @staticmethod
    def _shape(size):
        if len(size) == 1 and not isinstance(size[0], int):   # a torch.Size, tuple or list
            return tuple(size[0])
        return tuple(size)

    def _device_ok(self, device):
        return device is not None and self._t.device(device).type == "cuda"

    def empty(self, *size, dtype=None, device=None, **kw):
        if not self._device_ok(device) or kw.get("pin_memory"):
            return self._t.empty(*size, dtype=dtype, device=device, **kw)
        return self._a.make(self._shape(size), dtype or self._t.get_default_dtype(), device)

    def zeros(self, *size, dtype=None, device=None, **kw):
        if not self._device_ok(device):
            return self._t.zeros(*size, dtype=dtype, device=device, **kw)
        return self._a.make(self._shape(size), dtype or self._t.get_default_dtype(), device, fill=0)

    def empty_like(self, t, dtype=None, device=None, **kw):
        dev = device if device is not None else t.device
        if not self._device_ok(dev) or kw:
            return self._t.empty_like(t, dtype=dtype, device=device, **kw)
        return self._a.make(tuple(t.shape), dtype or t.dtype, dev)
