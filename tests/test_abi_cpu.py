"""CPU checks of the C ABI: the library loads, exports every function that
include/ofrl.h declares, the ctypes mirrors match the C struct layouts, and
host-side argument checks answer without touching a GPU."""
import ctypes as C
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ofrl.h")
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    from offline_rl_step_gb300 import _abi, build
    build.build()
    return _abi.load()


def declared_functions():
    text = "\n".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[\w\s\*]+?\b(ofrl_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("ofrl_create", "ofrl_destroy", "ofrl_poll_status", "ofrl_status_string", "ofrl_her_relabel",
                 "ofrl_iql_value_fwd_bwd", "ofrl_expectile_loss", "ofrl_adv_weighted_policy",
                 "ofrl_budgeted_clip_saxpy", "ofrl_adam_step", "ofrl_train_step", "ofrl_workspace_bytes"):
        assert want in names


def test_library_exports_every_declared_function(lib):
    from offline_rl_step_gb300 import _abi
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in ofrl.h but not exported"
        assert name in _abi.SIGNATURES, f"{name} has no ctypes signature"


PROBE = r"""
#include <stddef.h>
#include <stdio.h>
#include "ofrl.h"
#define P(T, F) printf(#T "." #F " %zu\n", offsetof(T, F));
int main(void) {
  printf("ofrl_replay %zu\nofrl_her_cfg %zu\nofrl_batch %zu\nofrl_vshape %zu\nofrl_vnet %zu\nofrl_opt %zu\n",
         sizeof(ofrl_replay), sizeof(ofrl_her_cfg), sizeof(ofrl_batch), sizeof(ofrl_vshape),
         sizeof(ofrl_vnet), sizeof(ofrl_opt));
  P(ofrl_replay, episode_ends) P(ofrl_replay, capacity) P(ofrl_replay, num_episodes) P(ofrl_replay, goal_dim)
  P(ofrl_her_cfg, goal_threshold) P(ofrl_her_cfg, seed)
  P(ofrl_batch, donor_idx) P(ofrl_batch, stride)
  P(ofrl_vnet, t) P(ofrl_vnet, tau) P(ofrl_vnet, target) P(ofrl_vnet, polyak)
  P(ofrl_opt, beta) P(ofrl_opt, budget) P(ofrl_opt, alpha) P(ofrl_opt, weight_clamp_max_abs) P(ofrl_opt, sanitize_sources)
  return 0;
}
"""


def test_struct_layouts_match_the_header(tmp_path):
    from offline_rl_step_gb300 import _abi
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "probe.c"
    src.write_text(PROBE)
    exe = tmp_path / "probe"
    subprocess.run([cc, "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    out = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    mirrors = {"ofrl_replay": _abi.Replay, "ofrl_her_cfg": _abi.HerCfg, "ofrl_batch": _abi.Batch,
               "ofrl_vshape": _abi.VShape, "ofrl_vnet": _abi.VNet, "ofrl_opt": _abi.Opt}
    for cname, py in mirrors.items():
        assert int(out[cname]) == C.sizeof(py), cname
    for key, val in out.items():
        if "." in key:
            cname, field = key.split(".")
            assert getattr(mirrors[cname], field).offset == int(val), key


def test_host_side_answers(lib):
    from offline_rl_step_gb300 import _abi
    assert lib.ofrl_status_string(0) == b"OFRL_OK"
    assert b"EINVAL" in lib.ofrl_status_string(-1)
    ok = _abi.VShape(50, 128, 5, 0)
    assert lib.ofrl_workspace_bytes(C.byref(ok), 16384, 1) > 16384 // 128 * 23169 * 4
    assert lib.ofrl_workspace_bytes(C.byref(_abi.VShape(50, 96, 5, 0)), 16384, 1) == -1
    assert lib.ofrl_workspace_bytes(C.byref(ok), 16384, 3) == -1
    # a null context is refused before any CUDA call
    assert lib.ofrl_her_relabel(None, None, None, 0, None, None) == _abi.EINVAL
    assert lib.ofrl_train_step(None, None, None, 0, None, None, None, 0, None, None, 0,
                               None, None, None, None, None, None, None) == _abi.EINVAL
    out = C.c_void_p(1)
    assert lib.ofrl_create(C.byref(_abi.VShape(0, 128, 5, 0)), 16, 1, C.byref(out)) == _abi.EINVAL
    assert out.value is None


def test_binding_refuses_without_library(tmp_path):
    from offline_rl_step_gb300 import _abi
    saved = _abi._LIB
    try:
        _abi._LIB = None
        with pytest.raises(RuntimeError, match="not built"):
            _abi.load(str(tmp_path / "missing.so"))
    finally:
        _abi._LIB = saved
