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
