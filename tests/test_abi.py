"""The C-ABI library loads, exports every entry point include/ep.h declares and
rejects bad arguments on the host before touching the GPU. CPU only: no call
here reaches a kernel launch or a CUDA API call."""
import ctypes
import pathlib
import re

import pytest

ROOT = pathlib.Path(__file__).resolve().parents[1]
HEADERS = sorted((ROOT / "include").glob("*.h"))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__._cuda_build_module().build()
    import combine_router_softmax_gb300 as m

    return m


def declared_functions():
    names = []
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_]\w*\s*\*?\s*(ep_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_headers_declare_the_path():
    names = declared_functions()
    for required in ("ep_route", "ep_layout", "ep_dispatch", "ep_combine"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(str(lib.LIB_PATH))
    missing = [n for n in declared_functions() if not hasattr(so, n)]
    assert not missing, f"declared but not exported: {missing}"
    assert set(lib.EXPORTS) == set(declared_functions())


def test_struct_layout(lib):
    assert ctypes.sizeof(lib.EpConfig) == 12 * 4
    assert ctypes.sizeof(lib.EpChunk) == 5 * 4


def test_status_strings(lib):
    for s in range(5):
        assert lib.ep_status_string(s).startswith("EP_")
    assert lib.ep_status_string(99) == "EP_ERR_UNKNOWN"
    assert lib.ep_version() >= 100


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails validation first


def _cfg(lib, **kw):
    base = dict(T=64, H=256, E=16, R=4, k=2, num_workers=8)
    base.update(kw)
    return lib.EpConfig.make(**base)


@pytest.mark.parametrize("bad,expect", [
    (dict(E=15), "INVALID"),            # E % R
    (dict(k=17), "INVALID"),            # k > E
    (dict(T=-1), "INVALID"),
    (dict(n_groups=3), "INVALID"),      # E % n_groups
    (dict(n_groups=4, topk_groups=5), "INVALID"),
    (dict(n_groups=8, topk_groups=1, k=3), "INVALID"),  # 1 group of 2 < k
    (dict(renormalize=2), "INVALID"),
    (dict(E=2048, R=4), "UNSUPPORTED"),
    (dict(E=64, k=33), "UNSUPPORTED"),
    (dict(E=64, n_groups=64, topk_groups=2), "UNSUPPORTED"),
    (dict(T=2**30, k=4), "INVALID"),    # T k > INT32_MAX
])
def test_config_validation(lib, bad, expect):
    cfg = _cfg(lib, **bad)
    rc = lib._lib.ep_route(ctypes.byref(cfg), FAKE, FAKE, FAKE, None)
    assert rc == (lib.EP_ERR_INVALID_ARG if expect == "INVALID" else lib.EP_ERR_UNSUPPORTED)


def test_null_and_shape_errors(lib):
    L = lib._lib
    assert L.ep_route(None, FAKE, FAKE, FAKE, None) == lib.EP_ERR_INVALID_ARG
    cfg = _cfg(lib)
    assert L.ep_route(ctypes.byref(cfg), None, FAKE, FAKE, None) == lib.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(ctypes.byref(_cfg(lib, H=12)), FAKE, FAKE, FAKE, FAKE, None) == lib.EP_ERR_UNSUPPORTED
    assert L.ep_dispatch(ctypes.byref(_cfg(lib, H=0)), FAKE, FAKE, FAKE, FAKE, None) == lib.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(ctypes.byref(cfg), ctypes.c_void_p(0x10008), FAKE, FAKE, FAKE, None) == lib.EP_ERR_INVALID_ARG
    assert L.ep_combine(ctypes.byref(cfg), FAKE, FAKE, FAKE, ctypes.c_void_p(0x10004), None) == lib.EP_ERR_INVALID_ARG
    assert L.ep_combine(ctypes.byref(cfg), FAKE, None, FAKE, FAKE, None) == lib.EP_ERR_INVALID_ARG


def test_pod_tier_capacity_and_validation(lib):
    """With a pod tier the schedule has three hop classes: capacity 3 W + R;
    ranks_per_pod must be a non-negative multiple of ranks_per_node."""
    assert lib.ep_schedule_capacity(_cfg(lib, ranks_per_node=2, ranks_per_pod=4)) == 3 * 8 + 4
    assert lib.ep_schedule_capacity(_cfg(lib, ranks_per_node=2, ranks_per_pod=0)) == 2 * 8 + 4
    n = ctypes.c_int32(0)
    for bad in (dict(ranks_per_node=2, ranks_per_pod=3), dict(ranks_per_pod=-16)):
        rc = lib._lib.ep_schedule_capacity(ctypes.byref(_cfg(lib, **bad)), ctypes.byref(n))
        assert rc == lib.EP_ERR_INVALID_ARG


def test_layout_capacity_and_workspace_errors(lib):
    L = lib._lib
    cfg = _cfg(lib, T=1000)
    cap = lib.ep_schedule_capacity(cfg)
    assert cap == 2 * 8 + 4
    ws = lib.ep_layout_workspace_size(cfg)
    assert ws >= 16 * 4 * 4 and ws % 256 == 0  # 4 layout CTAs x 16 experts
    args = [FAKE] * 6
    # chunk table too small
    rc = L.ep_layout(ctypes.byref(cfg), *args, FAKE, ctypes.c_int32(cap - 1), FAKE, FAKE, FAKE,
                     ctypes.c_size_t(ws), None)
    assert rc == lib.EP_ERR_CAPACITY
    # workspace too small
    rc = L.ep_layout(ctypes.byref(cfg), *args, FAKE, ctypes.c_int32(cap), FAKE, FAKE, FAKE,
                     ctypes.c_size_t(ws - 256), None)
    assert rc == lib.EP_ERR_CAPACITY
    # workspace not 256-byte aligned
    rc = L.ep_layout(ctypes.byref(cfg), *args, FAKE, ctypes.c_int32(cap), FAKE, FAKE, ctypes.c_void_p(0x10010),
                     ctypes.c_size_t(ws), None)
    assert rc == lib.EP_ERR_INVALID_ARG
    # self_rank outside [0, R)
    rc = L.ep_layout(ctypes.byref(_cfg(lib, self_rank=4)), *args, FAKE, ctypes.c_int32(cap), FAKE, FAKE, FAKE,
                     ctypes.c_size_t(ws), None)
    assert rc == lib.EP_ERR_INVALID_ARG


def test_T0_calls_enqueue_nothing(lib):
    cfg = _cfg(lib, T=0)
    L = lib._lib
    assert L.ep_route(ctypes.byref(cfg), None, None, None, None) == lib.EP_OK
    assert L.ep_dispatch(ctypes.byref(cfg), None, None, None, None, None) == lib.EP_OK
    assert L.ep_combine(ctypes.byref(cfg), None, None, None, None, None) == lib.EP_OK
    assert lib.ep_layout_workspace_size(cfg) == 0


def test_binding_rejects_cpu_tensors(lib):
    import torch

    cfg = _cfg(lib, T=4, E=8, R=4)
    with pytest.raises(ValueError):
        lib.ep_route(cfg, torch.zeros((4, 8)), torch.zeros((4, 2), dtype=torch.int32), torch.zeros((4, 2)))
    with pytest.raises(TypeError):
        lib.ep_route(cfg, torch.zeros((4, 8), dtype=torch.float64), torch.zeros((4, 2), dtype=torch.int32),
                     torch.zeros((4, 2)))
