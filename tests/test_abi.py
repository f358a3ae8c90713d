"""The C-ABI library builds, loads and exports every symbol the header
declares; host-side argument checks work without a GPU (no kernel runs)."""
import ctypes
import os
import re
import shutil

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ep.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def ep():
    from combine_get_dispatch_notify_gb300 import build, ep as binding
    build.build()
    binding.lib()
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ep_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(ep):
    names = declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(ep.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ep.h but not exported"
    assert sorted(ep.exported_symbols()) == names


def declared_arity():
    """Parameter count of every function the header declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(ep_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_arity_matches_header(ep):
    arity = declared_arity()
    lib = ep.lib()
    for name in ep.exported_symbols():
        assert len(getattr(lib, name).argtypes) == arity[name], name


def test_library_links_against_the_shared_cuda_runtime(ep):
    with open("/proc/self/maps") as f:
        maps = f.read()
    assert "libep_gb300.so" in maps


def test_shape_rules(ep):
    S = ep.EpShape.make
    ok = [S(1, 5, 1, 1, 8, 1), S(2, 128, 2, 16, 256, 2), S(16, 128, 8, 256, 7168, 8),
          S(32, 16384, 8, 256, 7168, 32), S(3, 0, 2, 9, 72, 5), S(8, 10, 32, 8192, 8, 4096)]
    bad = [S(0, 5, 1, 1, 8, 1), S(12, 5, 1, 12, 8, 1), S(40, 5, 1, 40, 8, 1), S(2, 5, 0, 2, 8, 1),
           S(2, 5, 33, 2, 8, 1), S(4, 5, 2, 6, 8, 1), S(4, 5, 2, 2, 8, 1), S(2, 5, 2, 4, 12, 1),
           S(2, 5, 2, 4, 8, 0), S(2, -1, 2, 4, 8, 1), S(32, 1 << 25, 8, 256, 8, 1),
           ep.EpShape(2, 5, 2, 4, 8, 1, 0), S(2, 5, 2, 4, 8, 4097)]
    for s in ok:
        assert ep.ep_check_shape(s) == ep.EP_OK, tuple(getattr(s, f) for f, _ in s._fields_)
    for s in bad:
        assert ep.ep_check_shape(s) == ep.EP_ERR_INVALID_ARG, tuple(getattr(s, f) for f, _ in s._fields_)


def test_nodes_and_workspace(ep):
    S = ep.EpShape.make
    assert ep.ep_num_nodes(S(4, 8, 2, 8, 8, 2)) == 1
    assert ep.ep_num_nodes(S(8, 8, 2, 8, 8, 2)) == 1
    assert ep.ep_num_nodes(S(16, 8, 2, 16, 8, 2)) == 2
    assert ep.ep_num_nodes(S(32, 8, 2, 32, 8, 2)) == 4
    assert ep.ep_num_nodes(S(12, 8, 2, 12, 8, 2)) == -1
    # one 8-byte lookback word per (block, rank or node), plus a header
    s = S(16, 128, 8, 256, 7168, 8)
    assert ep.ep_notify_workspace_bytes(s) == 256 + 16 * 8 * (16 + 2) * 8
    assert ep.ep_notify_workspace_bytes(S(12, 8, 2, 12, 8, 2)) == 0


def test_status_strings(ep):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert ep.ep_status_string(code) and ep.ep_status_string(code) != "unknown status"
    assert ep.ep_status_string(7) == "unknown status"


def test_invalid_calls_return_before_touching_the_device(ep):
    """Bad shapes and NULL / misaligned pointers are refused on the host."""
    vp = ctypes.c_void_p
    good = ep.EpShape.make(2, 4, 2, 4, 8, 2)
    badshape = ep.EpShape.make(12, 4, 2, 12, 8, 2)
    fake = vp(1 << 20)        # aligned, never dereferenced: the call must fail first
    odd = vp((1 << 20) + 4)   # misaligned for 16-byte arrays
    L = ep.lib()
    assert L.ep_get_dispatch_layout(ctypes.byref(badshape), fake, fake, fake, fake, fake, fake,
                                    vp(0)) == ep.EP_ERR_INVALID_ARG
    assert L.ep_get_dispatch_layout(ctypes.byref(good), odd, fake, fake, fake, fake, fake,
                                    vp(0)) == ep.EP_ERR_INVALID_ARG
    assert L.ep_get_dispatch_layout(ctypes.byref(good), vp(None), fake, fake, fake, fake, fake,
                                    vp(0)) == ep.EP_ERR_INVALID_ARG
    nul = vp(None)  # sched: optional
    assert L.ep_dispatch(ctypes.byref(good), fake, fake, fake, fake, fake, ctypes.c_int64(-1), fake,
                         fake, fake, fake, fake, nul, vp(0)) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(ctypes.byref(good), odd, fake, fake, fake, fake, ctypes.c_int64(8), fake,
                         fake, fake, fake, fake, nul, vp(0)) == ep.EP_ERR_INVALID_ARG
    # top-k arrays are all-or-none (none = cached mode)
    assert L.ep_dispatch(ctypes.byref(good), fake, fake, vp(None), fake, fake, ctypes.c_int64(8), fake,
                         fake, fake, fake, fake, nul, vp(0)) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(ctypes.byref(good), fake, fake, fake, fake, fake, ctypes.c_int64(8), fake,
                         vp(None), vp(None), fake, fake, nul, vp(0)) == ep.EP_ERR_INVALID_ARG
    # a misaligned sched word is refused
    assert L.ep_dispatch(ctypes.byref(good), fake, fake, fake, fake, fake, ctypes.c_int64(8), fake,
                         fake, fake, fake, fake, odd, vp(0)) == ep.EP_ERR_INVALID_ARG
    assert L.ep_combine(ctypes.byref(good), vp(None), vp(None), 4, fake, fake, fake, vp(None), fake,
                        vp(0)) == ep.EP_ERR_INVALID_ARG  # y missing
    assert L.ep_combine(ctypes.byref(good), fake, vp(None), 4, fake, fake, fake, fake, fake,
                        vp(0)) == ep.EP_ERR_INVALID_ARG  # combined_w without y_w
    assert L.ep_combine(ctypes.byref(good), fake, fake, -1, fake, fake, fake, fake, fake,
                        vp(0)) == ep.EP_ERR_INVALID_ARG  # negative y_rows
    args = [fake] * 16
    assert L.ep_notify_dispatch(ctypes.byref(good), *args, ctypes.c_size_t(8), fake, vp(None),
                                vp(0)) == ep.EP_ERR_INVALID_ARG  # workspace too small
    assert L.ep_debug_notify_dispatch_stall(ctypes.byref(good), *args, ctypes.c_size_t(1 << 20), fake,
                                            0, 0, vp(0)) == ep.EP_ERR_INVALID_ARG  # zero wait limit


def test_binding_refuses_cpu_tensors(ep):
    s = ep.EpShape.make(2, 4, 2, 4, 8, 2)
    t = torch.zeros(2, 4, 2, dtype=torch.int64)
    with pytest.raises(ValueError):
        ep.ep_get_dispatch_layout(s, t, None, None, None, None, None)


C_CONSUMER = r"""
#include <stdio.h>
#include "ep.h"

int main(void) {
    ep_shape_t ok = {16, 128, 8, 256, 7168, 8, 1};
    ep_shape_t bad = {12, 128, 8, 256, 7168, 8, 1};  /* 12 ranks: not a multiple of 8 */
    printf("%d %d %d %zu %s\n", (int)ep_check_shape(&ok), (int)ep_check_shape(&bad), (int)ep_num_nodes(&ok),
           ep_notify_workspace_bytes(&ok), ep_status_string(EP_ERR_CAPACITY));
    return 0;
}
"""


def test_c_consumer_compiles_links_and_runs(ep, tmp_path):
    """A plain C11 program includes ep.h, links libep_gb300.so and calls its
    host-only entry points (no device work)."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    src = tmp_path / "consumer.c"
    src.write_text(C_CONSUMER)
    exe = tmp_path / "consumer"
    lib_dir = os.path.dirname(ep.LIB_PATH)
    cmd = [gcc, "-std=c11", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
           str(src), "-o", str(exe), "-L", lib_dir, "-lep_gb300", f"-Wl,-rpath,{lib_dir}"]
    import subprocess
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    ok, bad, nodes, ws, msg = out.stdout.split(" ", 4)
    assert int(ok) == ep.EP_OK and int(bad) == ep.EP_ERR_INVALID_ARG and int(nodes) == 2
    assert int(ws) == 256 + 16 * 8 * (16 + 2) * 8
    assert msg.strip() == "receive capacity exceeded"


def test_layout_notify_workspace_bytes_follow_the_documented_formula(ep):
    """Host-only: 256-byte header + 1 MiB + 32 KiB of expert counters + 8 (R+N)
    bytes per tile + 8 R (R+N), with tiles of 512 tokens (fewer when T is
    smaller, larger beyond 16384 tiles); 0 for an invalid shape."""
    def want(R, T):
        N = 1 if R <= 8 else R // 8
        V = R + N
        tt = 256 if T >= 256 else max(32, -(-T // 32) * 32)
        while tt < 8192 and R * -(-T // tt) > 16384:
            tt *= 2
        tiles = R * (-(-T // tt) if T > 0 else 1)
        return 256 + (2 << 20) + (64 << 10) + (18 << 10) + 8 * V * tiles

    for R, T in [(1, 0), (2, 1), (3, 41), (8, 4096), (16, 8192), (32, 16384), (32, 20000), (16, 300),
                 (32, 2 ** 25 - 1)]:  # R*T just under 2^30
        sh = ep.EpShape.make(R, T, 8, R * 8, 7168, 24)  # E % R == 0
        assert ep.ep_layout_notify_workspace_bytes(sh) == want(R, T), (R, T)
    bad = ep.EpShape.make(12, 16, 8, 256, 7168, 24)  # R > 8 and not whole nodes
    assert ep.ep_layout_notify_workspace_bytes(bad) == 0
