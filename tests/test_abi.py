"""The C-ABI library loads, exports every entry point include/ep.h declares and
rejects bad arguments on the host before touching the GPU. CPU only: no call
here reaches a kernel launch or a CUDA API call."""
import ctypes
import os
import pathlib
import re
import shutil
import subprocess
import sys

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


@pytest.mark.parametrize("E,R,k", [(8, 4, 2), (256, 32, 8), (128, 16, 8), (96, 6, 12), (1024, 32, 32)])
def test_layout_workspace_within_the_documented_bound(lib, E, R, k):
    """include/ep.h: the layout's scratch is at most 4 E max(ceil(T / 256), 64)
    + 512 bytes and at least the three-kernel layout's 4 E ceil(T / 256)."""
    for T in (1, 63, 64, 1000, 2049, 4096, 16385, 32768, 32769, 65536, 100000, 262144):
        n = lib.ep_layout_workspace_size(lib.EpConfig.make(T=T, H=64, E=E, R=R, k=k, num_workers=8))
        blocks = (T + 255) // 256
        assert 4 * E * blocks <= n <= 4 * E * max(blocks, 64) + 512, (T, n)


def test_static_layout_limit_is_the_documented_one(lib):
    """E = 256 fits ep_layout_static's 1 MiB array up to T = 262144 and no further."""
    def ws(T):
        return lib.ep_layout_workspace_size(lib.EpConfig.make(T=T, H=64, E=256, R=32, k=8, num_workers=8))

    assert ws(262144) <= lib.EP_LAYOUT_STATIC_SCRATCH_BYTES < ws(262145)


def test_layout_capacity_and_workspace_errors(lib):
    L = lib._lib
    cfg = _cfg(lib, T=1000)
    cap = lib.ep_schedule_capacity(cfg)
    assert cap == 2 * 8 + 4
    ws = lib.ep_layout_workspace_size(cfg)
    assert ws >= 16 * 4 * 4 and ws % 256 == 0  # at least the three-kernel layout's 4 CTAs x 16 experts
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


U = ctypes.c_void_p(0x10008)  # 8-byte aligned, not 16


def test_tff_framed_bytes(lib):
    """T k ceil(2H / 480) blocks of 512 bytes."""
    n = ctypes.c_size_t(0)
    for T, H, k, blocks in ((64, 256, 2, 2), (3, 7168, 8, 30), (5, 240, 2, 1), (1, 8, 1, 1), (2, 24576, 4, 103)):
        cfg = _cfg(lib, T=T, H=H, k=k)
        assert lib._lib.ep_tff_framed_bytes(ctypes.byref(cfg), ctypes.byref(n)) == lib.EP_OK
        assert n.value == T * k * blocks * 512
    assert lib._lib.ep_tff_framed_bytes(ctypes.byref(_cfg(lib, H=12)), ctypes.byref(n)) == lib.EP_ERR_UNSUPPORTED


def test_added_entry_points_reject_bad_arguments(lib):
    L = lib._lib
    cfg = _cfg(lib, H=1024, k=4)
    bad = lib.EP_ERR_INVALID_ARG
    # TFF codec: null or misaligned buffers
    assert L.ep_tff_encode(ctypes.byref(cfg), None, FAKE, 1, None) == bad
    assert L.ep_tff_encode(ctypes.byref(cfg), U, FAKE, 1, None) == bad
    assert L.ep_tff_decode(ctypes.byref(cfg), FAKE, 1, FAKE, None, None) == bad
    assert L.ep_tff_decode(ctypes.byref(cfg), FAKE, 1, FAKE, ctypes.c_void_p(0x10002), None) == bad
    # sentinel arm / expert scale
    assert L.ep_sentinel_arm(ctypes.byref(cfg), None, None) == bad
    assert L.ep_sentinel_arm(ctypes.byref(cfg), U, None) == bad
    assert L.ep_expert_scale(ctypes.byref(cfg), FAKE, None, FAKE, FAKE, None) == bad
    # producer/consumer handoffs: null tables, misaligned slot, unsupported shapes
    args = [FAKE] * 10
    assert L.ep_dispatch_expert_sp(ctypes.byref(cfg), *args[:5], None, *args[6:], None) == bad
    assert L.ep_dispatch_expert_sp(ctypes.byref(cfg), FAKE, U, *args[2:], None) == bad
    assert L.ep_dispatch_expert_sp(ctypes.byref(_cfg(lib, H=1024, k=2)), *args, None) == lib.EP_ERR_UNSUPPORTED
    assert L.ep_dispatch_expert_sp(ctypes.byref(_cfg(lib, H=256, k=4)), *args, None) == lib.EP_ERR_UNSUPPORTED
    assert L.ep_dispatch_expert_sw(ctypes.byref(cfg), *args, None, 1, None) == bad
    assert L.ep_dispatch_expert_sw(ctypes.byref(cfg), *args, ctypes.c_void_p(0x10002), 1, None) == bad
    assert L.ep_dispatch_expert_sw(ctypes.byref(_cfg(lib, H=1024, k=6)), *args, FAKE, 1, None) == \
        lib.EP_ERR_UNSUPPORTED
    # schedule-driven dispatch: null pointers, misaligned cta_ns, rows above 48 KiB
    assert L.ep_dispatch_scheduled(ctypes.byref(cfg), None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == bad
    assert L.ep_dispatch_scheduled(ctypes.byref(cfg), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                   ctypes.c_void_p(0x10004), None) == bad
    big = _cfg(lib, H=32768, k=4)
    assert L.ep_dispatch_scheduled(ctypes.byref(big), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == \
        lib.EP_ERR_UNSUPPORTED


def test_header_is_plain_c(lib, tmp_path):
    """include/ep.h compiles as C11 with every warning an error, and a C program
    that names every entry point links against the library and calls the
    host-only ones (no GPU needed)."""
    gcc = shutil.which("gcc")
    cuda_inc = pathlib.Path(os.environ.get("CUDA_HOME", "/usr/local/cuda")) / "include"
    if not gcc or not (cuda_inc / "cuda_runtime_api.h").exists():
        pytest.skip("gcc or the CUDA headers are not available")
    names = declared_functions()
    table = ",\n    ".join(f"(fn_t){n}" for n in names)
    src = tmp_path / "use_ep.c"
    src.write_text(f"""#include <stdio.h>
#include "ep.h"

typedef void (*fn_t)(void);
static const fn_t entry_points[] = {{
    {table}
}};

int main(void) {{
    ep_config c = {{1000, 64, 16, 4, 2, 1, 1, 1, 2, 0, 8, 0}};
    size_t ws = 0;
    int32_t cap = 0;
    ep_status a = ep_layout_workspace_size(&c, &ws);
    ep_status b = ep_schedule_capacity(&c, &cap);
    printf("%d %d %d %zu %d %s\\n", (int)(sizeof entry_points / sizeof entry_points[0]), (int)a, (int)b, ws,
           (int)cap, ep_status_string(EP_ERR_CAPACITY));
    return 0;
}}
""")
    exe = tmp_path / "use_ep"
    libdir = pathlib.Path(lib.__file__).resolve().parent
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", f"-I{ROOT / 'include'}",
                        f"-I{cuda_inc}", str(src), "-o", str(exe), f"-L{libdir}", "-lep_gb300",
                        f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split(maxsplit=5)
    cfg = lib.EpConfig.make(T=1000, H=64, E=16, R=4, k=2, ranks_per_node=2, num_workers=8)
    assert int(out[0]) == len(names)
    assert out[1] == out[2] == "0"
    assert int(out[3]) == lib.ep_layout_workspace_size(cfg)
    assert int(out[4]) == lib.ep_schedule_capacity(cfg) == 2 * 8 + 4
    assert out[5].startswith("EP_ERR_CAPACITY")


def test_package_refuses_to_import_without_the_library(tmp_path):
    """With the CUDA library missing, importing the package fails loudly: there is
    no CPU or PyTorch fallback to land on."""
    pkg = tmp_path / "combine_router_softmax_gb300"
    pkg.mkdir()
    shutil.copy(ROOT / "combine_router_softmax_gb300" / "__init__.py", pkg / "__init__.py")
    env = dict(os.environ, PYTHONPATH=str(tmp_path))
    r = subprocess.run([sys.executable, "-c", "import combine_router_softmax_gb300"], cwd=tmp_path, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "There is no fallback path" in r.stderr
