"""The debug build (MOE_CHECKS=1) on the host: it is built beside the default
library, the binding selects it from the environment, it reports its build
flags, and it refuses bad configs like the default build (no GPU needed)."""
import ctypes
import json
import os
import subprocess
import sys

import pytest

from quantized_moe_decode_gemv_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROBE = r"""
import ctypes, json
import quantized_moe_decode_gemv_gb300 as pkg
from quantized_moe_decode_gemv_gb300 import _capi
lib = pkg.load_library()
cfg = pkg.MoEConfig(hidden=512, n_experts=16, top_k=40, expert_ffn=256).to_c()
print(json.dumps({"lib": _capi.LIB_NAME, "flags": lib.moe_build_flags(),
                  "abi": lib.moe_abi_version(),
                  "refusal": _capi.STATUS_NAMES[lib.moe_layer_validate(ctypes.byref(cfg), None)],
                  "index_name": lib.moe_status_string(11).decode()}))
"""


def _probe(checks: bool):
    env = dict(os.environ)
    env.pop("MOE_CHECKS", None)
    if checks:
        env["MOE_CHECKS"] = "1"
    r = subprocess.run([sys.executable, "-c", PROBE], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_both_builds_exist():
    for lib in (B.LIB, B.LIB_CHECKS):
        if not os.path.exists(lib):
            pytest.fail(f"{os.path.basename(lib)} is not built; run __graft_entry__.build()")


def test_debug_build_is_selected_and_flagged():
    plain, checks = _probe(False), _probe(True)
    assert plain["lib"] == "libmoe_gb300.so" and plain["flags"] == 0
    assert checks["lib"] == "libmoe_gb300_checks.so"
    assert checks["flags"] == 3   # MOE_BUILD_CHECKS | MOE_BUILD_NVTX_DEFAULT
    for r in (plain, checks):
        assert r["abi"] == 4
        assert r["refusal"] == "MOE_ERR_TOPK_GT_E"
        assert r["index_name"] == "MOE_ERR_INDEX"


def test_debug_build_compiles_the_checks():
    """The check macro is off by default and on in the debug objects: the
    default build's flags word is a compile-time constant of MOE_CHECKS."""
    src = open(os.path.join(B.CSRC, "moe_kernels.cuh")).read()
    assert "#ifndef MOE_CHECKS\n#define MOE_CHECKS 0" in src
    assert any("-DMOE_CHECKS=1" in v[2] for v in B.VARIANTS)
