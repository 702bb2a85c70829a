"""Host-only checks of the C ABI: the library builds and loads, exports every
entry point include/*.h declares, and rejects bad arguments on the host
before anything reaches a GPU (no call here launches a kernel)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    import moe_routed_expert_gb300 as M
    return M.load()


def declared_functions():
    names = []
    for h in HEADERS:
        names += re.findall(r"^MOE_API\s+[\w\s\*]+?\b(\w+)\s*\(", open(h).read(), flags=re.M)
    return names


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    for n in ("gmm_forward", "gmm_backward", "moe_permute", "moe_unpermute", "moe_layer_forward",
              "moe_layer_backward", "moe_unpermute_backward", "moe_permute_backward", "moe_swiglu_backward",
              "moe_mx_quantize", "moe_permute_mx", "gmm_forward_mx", "moe_layer_forward_mx"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import subprocess
    from moe_routed_expert_gb300 import _abi
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.lib_path()], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(lib, n)
    # nothing else leaks out of the library's C++ internals
    assert all(not e.startswith("_ZN3moe") for e in exported)
    assert set(_abi.SIGNATURES) == set(declared_functions())


def test_bounds_checking_build_exports_the_same_symbols():
    """The bounds-checking variant (-DMOE_BOUNDS_CHECK=1) builds from the same
    sources and exports the same entry points; the binding picks it only when
    MOE_GB300_BOUNDS_CHECK=1."""
    import subprocess
    from moe_routed_expert_gb300 import _abi, build
    path = build.build(bounds=True)
    assert path.endswith("libmoe_gb300_bounds.so") and path != build.LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert set(declared_functions()) <= exported
    assert all(not e.startswith("_ZN3moe") for e in exported)
    old = os.environ.get("MOE_GB300_BOUNDS_CHECK")
    try:
        os.environ["MOE_GB300_BOUNDS_CHECK"] = "1"
        assert _abi.bounds_checking() and _abi.lib_path() == path
        os.environ["MOE_GB300_BOUNDS_CHECK"] = "0"
        assert not _abi.bounds_checking() and _abi.lib_path() == build.LIB_PATH
    finally:
        if old is None:
            os.environ.pop("MOE_GB300_BOUNDS_CHECK", None)
        else:
            os.environ["MOE_GB300_BOUNDS_CHECK"] = old


def test_status_strings(lib):
    for code, name in {0: "MOE_OK", 1: "MOE_ERR_NULLPTR", 2: "MOE_ERR_INVALID", 3: "MOE_ERR_UNSUPPORTED",
                       4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE", 6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_BOUNDS"}.items():
        assert lib.moe_status_string(code).decode() == name


def test_workspace_sizes(lib):
    assert lib.gmm_workspace_size(8192, 1024, 2048, 8) == 256 + 256 * 6 * 256  # status + descriptor slots
    assert lib.moe_unpermute_workspace_size() == 256
    # permute: status block + per-chunk counts (1024 slots per chunk, int32 per expert)
    assert lib.moe_permute_workspace_size(4096, 8, 256) == 256 + 32 * 256 * 4
    assert lib.moe_permute_workspace_size(0, 8, 256) == 256
    T, H, I, E, k = 4096, 2048, 512, 256, 8
    n = lib.moe_layer_workspace_size(T, H, I, E, k)
    R = T * k
    assert n >= 256 + 256 * 6 * 256 + R * H * 2 * 2 + R * I * 2 + 2 * R * 4 + E * 8
    assert n % 256 == 0


FAKE = C.c_void_p(0x10000)   # never dereferenced: every call below fails its host checks first
MIS = C.c_void_p(0x10008)    # 8-byte aligned, not 16


def test_null_and_invalid_arguments_fail_on_the_host(lib):
    ws, nws = FAKE, 1 << 20
    # required pointer missing
    assert lib.gmm_forward(None, FAKE, FAKE, 64, 128, 256, 4, 0, 0.0, FAKE, None, ws, nws, None) == 1
    assert lib.moe_permute(FAKE, None, 4, 64, 2, 4, FAKE, FAKE, FAKE, FAKE, ws, nws, None) == 1
    assert lib.moe_permute(None, FAKE, 4, 64, 2, 4, FAKE, FAKE, FAKE, FAKE, ws, nws, None) == 1  # x without x_perm
    assert lib.moe_unpermute(FAKE, None, FAKE, 4, 64, 2, FAKE, ws, nws, None) == 1
    assert lib.moe_layer_backward(FAKE, FAKE, FAKE, FAKE, None, 4, 64, 128, 4, 2, 0.0, FAKE, FAKE, FAKE, FAKE,
                                  ws, nws, None) == 1
    # sizes
    assert lib.gmm_forward(FAKE, FAKE, FAKE, 64, 100, 256, 4, 0, 0.0, FAKE, None, ws, nws, None) == 3  # K % 64
    assert lib.gmm_forward(FAKE, FAKE, FAKE, 64, 128, 256, 2000, 0, 0.0, FAKE, None, ws, nws, None) == 3  # E
    assert lib.gmm_forward(FAKE, FAKE, FAKE, -1, 128, 256, 4, 0, 0.0, FAKE, None, ws, nws, None) == 2
    assert lib.gmm_forward(FAKE, FAKE, FAKE, 64, 128, 192, 4, 1, 0.0, FAKE, None, ws, nws, None) == 3  # SwiGLU N
    assert lib.gmm_forward(FAKE, FAKE, FAKE, 64, 128, 256, 4, 7, 0.0, FAKE, None, ws, nws, None) == 3  # epilogue
    assert lib.gmm_forward(FAKE, FAKE, FAKE, 64, 128, 256, 4, 1, -1.0, FAKE, None, ws, nws, None) == 2  # clip < 0
    assert lib.gmm_forward(FAKE, FAKE, FAKE, 64, 128, 256, 4, 1, float("nan"), FAKE, None, ws, nws, None) == 2
    assert lib.moe_permute(FAKE, FAKE, 4, 64, 5, 4, FAKE, FAKE, FAKE, FAKE, ws, nws, None) == 2  # k > E
    assert lib.moe_permute(FAKE, FAKE, 4, 64, 65, 100, FAKE, FAKE, FAKE, FAKE, ws, nws, None) == 3  # k > 64
    assert lib.moe_layer_forward(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 96, 4, 2, 0.0, FAKE, None, ws, nws,
                                 None) == 3  # I % 128
    # alignment and workspace size
    assert lib.gmm_forward(MIS, FAKE, FAKE, 64, 128, 256, 4, 0, 0.0, FAKE, None, ws, nws, None) == 2
    assert lib.gmm_forward(FAKE, FAKE, FAKE, 64, 128, 256, 4, 0, 0.0, FAKE, None, ws, 16, None) == 2
    assert lib.gmm_forward(FAKE, FAKE, FAKE, 64, 128, 256, 4, 0, 0.0, FAKE, None, None, nws, None) == 1
    assert lib.moe_permute(FAKE, FAKE, 4096, 64, 8, 256, FAKE, FAKE, FAKE, FAKE, ws, 256, None) == 2
    assert lib.moe_workspace_init(None, 256, None) == 1
    assert lib.moe_workspace_init(FAKE, 16, None) == 2


def test_fused_entry_points_check_their_arguments(lib):
    from moe_routed_expert_gb300 import _abi
    ws, nws = FAKE, 1 << 30
    act = _abi.MoeActivation(0, 0)
    a = C.byref(act)
    # gmm_forward_gather_act(x, sorted_flat, T, k, w, gl, M, K, N, E, act, flags, y, ws, n, s)
    g = lib.gmm_forward_gather_act
    assert g(FAKE, FAKE, 64, 2, FAKE, FAKE, 128, 256, 512, 4, None, 0, FAKE, ws, nws, None) == 1  # activation required
    assert g(FAKE, None, 64, 2, FAKE, FAKE, 128, 256, 512, 4, a, 0, FAKE, ws, nws, None) == 1
    assert g(FAKE, FAKE, 64, 2, FAKE, FAKE, 128, 256, 384, 4, a, 0, FAKE, ws, nws, None) == 3   # N % 256
    assert g(FAKE, FAKE, 64, 2, FAKE, FAKE, 128, 256, 512, 4, a, 4, FAKE, ws, nws, None) == 2   # flags
    assert g(FAKE, C.c_void_p(0x10002), 64, 2, FAKE, FAKE, 128, 256, 512, 4, a, 0, FAKE, ws, nws, None) == 2
    assert g(FAKE, FAKE, 64, 0, FAKE, FAKE, 128, 256, 512, 4, a, 0, FAKE, ws, nws, None) == 2   # k
    assert g(FAKE, FAKE, 64, 2, FAKE, FAKE, 128, 256, 512, 4, a, 0, FAKE, ws, 16, None) == 2   # workspace
    # gmm_forward_combine(a, w, gl, rmap, sflat, topk_w, T, k, M, K, N, E, flags, y, ws, n, s)
    c = lib.gmm_forward_combine
    assert c(FAKE, FAKE, FAKE, None, FAKE, FAKE, 64, 2, 128, 256, 512, 4, 0, FAKE, ws, nws, None) == 1
    assert c(None, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 2, 128, 256, 512, 4, 0, FAKE, ws, nws, None) == 1
    assert c(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 2, 128, 100, 512, 4, 0, FAKE, ws, nws, None) == 3  # K % 64
    assert c(MIS, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 2, 128, 256, 512, 4, 0, FAKE, ws, nws, None) == 2
    assert c(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 2, 128, 256, 512, 4, 0, FAKE, ws, 256, None) == 2
    # moe_expert_mlp_forward(x, sorted_flat, gl, w1, w2, T, H, I, E, k, act, a, y2, ws, n, s)
    f = lib.moe_expert_mlp_forward
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 64, 256, 128, 8, 2, None, FAKE, FAKE, ws, nws, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 64, 256, 96, 8, 2, a, FAKE, FAKE, ws, nws, None) == 3      # I % 128
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 64, 256, 128, 8, 9, a, FAKE, FAKE, ws, nws, None) == 2     # k > E
    assert f(FAKE, FAKE, FAKE, FAKE, MIS, 64, 256, 128, 8, 2, a, FAKE, FAKE, ws, nws, None) == 2
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 64, 256, 128, 8, 2, a, FAKE, FAKE, ws, 256, None) == 2     # workspace
    # status + one count per 128-row tile (T*k/128 + E), 256-byte aligned
    assert lib.moe_expert_mlp_workspace_size(4096, 8, 256) == 256 + (256 + 256) * 4
    # status + counts (ceil(N/256) int32, 256-byte aligned) + the [M, N] bf16 scratch
    assert lib.gmm_forward_combine_workspace_size(4096, 8, 32768, 2048) == 256 + 256 + 32768 * 2048 * 2
    assert lib.gmm_forward_combine_workspace_size(0, 8, 0, 2048) == 256


def test_activation_descriptor_checks(lib):
    """The (activation, activation_params) pair is checked on the host with the
    pages' rules: parameter counts per kind, clamp >= 0 and not NaN, finite
    alpha / beta, situglu's beta and linear_beta finite and > 0."""
    from moe_routed_expert_gb300 import _abi
    ws, nws = FAKE, 1 << 20

    def act(kind, *params):
        a = _abi.MoeActivation()
        a.kind, a.n_params = kind, len(params)
        for i, v in enumerate(params):
            a.params[i] = v
        return C.byref(a)

    def fwd(a):
        return lib.gmm_forward_act(FAKE, FAKE, FAKE, 64, 128, 256, 4, a, 0, FAKE, None, ws, nws, None)

    SW, STEP, OAI, SITU = 0, 1, 2, 3
    nan, inf = float("nan"), float("inf")
    assert lib.gmm_forward_act(None, FAKE, FAKE, 64, 128, 256, 4, None, 0, FAKE, None, ws, nws, None) == 1
    assert lib.gmm_forward_act(FAKE, FAKE, FAKE, 64, 128, 256, 4, None, 2, FAKE, None, ws, nws, None) == 2  # flags
    assert lib.gmm_forward_act(FAKE, FAKE, FAKE, 64, 128, 256, 4, None, 0, FAKE, FAKE, ws, nws, None) == 2  # h_save
    for bad in (act(SW, 1.0, 2.0), act(SW, -1.0), act(STEP, nan), act(OAI, 1.0), act(OAI, 1.0, inf, 1.0),
                act(OAI, 1.0, 1.0, nan), act(OAI, -2.0, 1.0, 1.0), act(SITU, 0.0), act(SITU, -1.0),
                act(SITU, 1.0, 0.0), act(SITU, inf), act(SITU, 1.0, 2.0, 3.0)):
        assert fwd(bad) == 2
    assert fwd(act(7)) == 3                                                   # unknown kind
    assert lib.gmm_forward_act(FAKE, FAKE, FAKE, 64, 128, 192, 4, act(SW), 0, FAKE, None, ws, nws, None) == 3  # N
    # valid descriptors get past the checks: a misaligned x is then what fails
    for good in (act(SW), act(SW, 0.0), act(STEP, 7.0), act(OAI), act(OAI, inf, 1.702, 1.0), act(SITU),
                 act(SITU, 2.0), act(SITU, 2.0, 3.0)):
        assert lib.gmm_forward_act(MIS, FAKE, FAKE, 64, 128, 256, 4, good, 1, FAKE, None, ws, nws, None) == 2
    assert lib.moe_activation_backward(FAKE, FAKE, 8, 64, act(SITU, -1.0), FAKE, ws, nws, None) == 2
    assert lib.gmm_backward_dx_act(FAKE, FAKE, FAKE, FAKE, 64, 128, 256, 4, None, 0, FAKE, ws, nws, None) == 1
    assert lib.moe_layer_forward_act(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 128, 4, 2, act(OAI, 1.0), 0, FAKE, None,
                                     ws, nws, None) == 2
    assert lib.moe_layer_forward_act(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 128, 4, 2, act(SW), 4, FAKE, None,
                                     ws, nws, None) == 2  # w_flags
    assert lib.gmm_backward_ex(FAKE, FAKE, FAKE, FAKE, 64, 128, 256, 4, 3, FAKE, FAKE, ws, nws, None) == 2


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    import moe_routed_expert_gb300 as M
    x = torch.zeros(64, 128, dtype=torch.bfloat16)
    w = torch.zeros(4, 128, 256, dtype=torch.bfloat16)
    gl = torch.tensor([16, 16, 0, 32])
    with pytest.raises((ValueError, RuntimeError)):
        M.gmm_forward(x, w, gl)


def test_wait_timeout_check_arguments(lib):
    assert lib.moe_check_wait_timeout(None, 256, 1000000, None) == 1
    assert lib.moe_check_wait_timeout(MIS, 256, 1000000, None) == 2
    assert lib.moe_check_wait_timeout(FAKE, 128, 1000000, None) == 2       # workspace too small
    assert lib.moe_check_wait_timeout(FAKE, 256, 10, None) == 2            # limit below 1 us
    assert lib.moe_check_wait_timeout(FAKE, 256, 20 * 10**9, None) == 2    # limit above 10 s


def test_bounds_check_arguments(lib):
    assert lib.moe_check_bounds(None, 256, None) == 1
    assert lib.moe_check_bounds(MIS, 256, None) == 2
    assert lib.moe_check_bounds(FAKE, 128, None) == 2                     # workspace too small


def test_mx_entry_points_check_their_arguments(lib):
    ws, nws = FAKE, 1 << 20
    a = _abi_act(0)
    assert lib.moe_mx_quantize_workspace_size() == 256
    assert lib.gmm_mx_workspace_size(64, 128, 256, 4) == 256
    T, H, I, E, k = 4096, 2048, 512, 256, 8
    R = T * k
    n = lib.moe_layer_mx_workspace_size(T, H, I, E, k)
    assert n >= 256 + R * H + R * H // 32 + R * I + R * I // 32 + R * H * 2 + 2 * R * 4 + E * 8
    # quantize: nulls, format, K % 32, alignment, zero rows is a no-op
    assert lib.moe_mx_quantize(None, 4, 64, 0, FAKE, FAKE, ws, nws, None) == 1
    assert lib.moe_mx_quantize(FAKE, 4, 64, 2, FAKE, FAKE, ws, nws, None) == 2
    assert lib.moe_mx_quantize(FAKE, 4, 48, 0, FAKE, FAKE, ws, nws, None) == 3
    assert lib.moe_mx_quantize(MIS, 4, 64, 0, FAKE, FAKE, ws, nws, None) == 2
    assert lib.moe_mx_quantize(None, 0, 64, 1, None, None, ws, nws, None) == 0
    # permute_mx
    assert lib.moe_permute_mx(FAKE, FAKE, 4, 64, 2, 4, 0, None, FAKE, FAKE, FAKE, FAKE, ws, nws, None) == 1
    assert lib.moe_permute_mx(FAKE, FAKE, 4, 64, 2, 4, 7, FAKE, FAKE, FAKE, FAKE, FAKE, ws, nws, None) == 2
    assert lib.moe_permute_mx(FAKE, FAKE, 4, 48, 2, 4, 0, FAKE, FAKE, FAKE, FAKE, FAKE, ws, nws, None) == 3
    assert lib.moe_permute_mx(FAKE, FAKE, 4, 64, 5, 4, 0, FAKE, FAKE, FAKE, FAKE, FAKE, ws, nws, None) == 2
    # gmm_forward_mx: plain needs y, activation needs a_q / a_scales; K and N multiples of 128
    gm = lambda M, K, N, act, y, aq, as_, h, x=FAKE: lib.gmm_forward_mx(x, FAKE, FAKE, FAKE, FAKE, M, K, N, 4, 0, 1,
                                                                         act, y, aq, as_, h, ws, nws, None)
    assert gm(64, 128, 256, None, None, None, None, None) == 1
    assert gm(64, 128, 256, a, FAKE, None, FAKE, None) == 1
    assert gm(64, 192, 256, None, FAKE, None, None, None) == 3
    assert gm(64, 128, 192, None, FAKE, None, None, None) == 3
    assert gm(64, 128, 384, a, None, FAKE, FAKE, None) == 3          # 2I must be a multiple of 256
    assert gm(64, 128, 256, None, FAKE, None, None, FAKE) == 2       # h_save without an activation
    assert gm(64, 128, 256, None, FAKE, None, None, None, x=MIS) == 2
    assert lib.gmm_forward_mx(FAKE, FAKE, FAKE, FAKE, FAKE, 64, 128, 256, 4, 3, 0, None, FAKE, None, None, None,
                              ws, nws, None) == 2                    # format
    assert gm(0, 128, 256, None, FAKE, None, None, None) == 0        # no rows: nothing to do
    # packed E2M1 operands (weights, or A4W4 tokens) want a 32-byte-aligned base
    e2m1 = lambda xf, x, w: lib.gmm_forward_mx(x, FAKE, w, FAKE, FAKE, 64, 128, 256, 4, xf, 5, None, FAKE, None,
                                               None, None, ws, nws, None)
    assert e2m1(0, FAKE, C.c_void_p(0x10010)) == 2
    assert e2m1(5, C.c_void_p(0x10010), FAKE) == 2
    assert e2m1(6, FAKE, FAKE) == 2                                  # E2M3 is not a format here
    # layer
    lay = lambda H, I, xf, act: lib.moe_layer_forward_mx(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, H, I, 4, 2,
                                                         xf, 0, act, FAKE, ws, nws, None)
    assert lay(128, 128, 0, None) == 1
    assert lay(128, 128, 9, a) == 2
    assert lay(192, 128, 0, a) == 3                                   # H % 128
    assert lay(128, 64, 0, a) == 3                                    # I % 128
    # A4W4: the packed tokens live in the workspace, which must then be 32-byte aligned
    assert lib.moe_layer_forward_mx(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 128, 128, 4, 2, 5, 5, a, FAKE,
                                    C.c_void_p(0x10010), 1 << 40, None) == 2


def _abi_act(kind, *params):
    from moe_routed_expert_gb300 import _abi
    x = _abi.MoeActivation()
    x.kind, x.n_params = kind, len(params)
    for i, v in enumerate(params):
        x.params[i] = v
    return C.byref(x)


def test_fp4_packing_layout():
    """E2M1 codes travel two per byte, element 2i in the low nibble (moe_mx.h)."""
    import numpy as np
    from workloads import pack_fp4, unpack_fp4
    c = np.arange(16, dtype=np.uint8).reshape(1, 16)
    p = pack_fp4(c)
    assert p.tolist() == [[0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE]]
    assert np.array_equal(unpack_fp4(p), c)
