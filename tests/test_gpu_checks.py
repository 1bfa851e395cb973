"""The debug build (MOE_CHECKS=1) on the GPU, in a child process that loads
libmoe_gb300_checks.so.

1. Clean runs: the tiny layer on the gemv path (1 and 3 rows) and the grouped
   path (16 rows) matches the oracle and leaves a clean status word.
2. Planted indices: MOE_DEBUG_BAD_INDEX makes the routing CTA write an expert
   id of E + 3 (1) or a pair id of T*k + 5 (2) into the route metadata of a
   one-row gemv forward.  Every consumer checks the index before it addresses
   memory, so the forward completes, the status call returns MOE_ERR_INDEX with
   the site, and the next clean forward matches the oracle again.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os
import numpy as np
import torch
import moe_inputs as mi
from tests import gpu_util as gu
import quantized_moe_decode_gemv_gb300 as pkg
from quantized_moe_decode_gemv_gb300 import _capi

lib = pkg.load_library()
assert _capi.LIB_NAME == "libmoe_gb300_checks.so" and lib.moe_build_flags() & 1
torch.cuda.set_device(0)
lay = gu.cached_layer("tiny", 0)
h = gu.build_layer(lay, 16)
res = {"clean": [], "planted": []}

def parity(T, path):
    x, _ = gu.margin_x(lay, T, seed=40 + T)
    h.set_path(path)
    got = gu.run_layer(h, x, lay.spec.act_dtype)
    gu.check_parity(got, gu.ora_forward(lay, x), what=f"checks build T={T} {path}")
    return _capi.STATUS_NAMES[h.device_status()]

for T, path in ((1, "gemv"), (3, "gemv"), (16, "grouped")):
    res["clean"].append([T, path, parity(T, path)])

x = gu.to_torch_x(gu.margin_x(lay, 1, seed=9)[0], lay.spec.act_dtype)
h.set_path("gemv")
for mode in ("1", "2"):
    os.environ["MOE_DEBUG_BAD_INDEX"] = mode
    h.forward(x)
    torch.cuda.synchronize()
    os.environ.pop("MOE_DEBUG_BAD_INDEX")
    st = _capi.STATUS_NAMES[h.device_status()]
    msg = lib.moe_layer_last_error(h.handle).decode()
    res["planted"].append([mode, st, msg, parity(1, "gemv")])
h.close()
print("RESULT " + json.dumps(res))
"""


def test_debug_build_clean_and_planted_indices():
    if not os.path.exists(os.path.join(ROOT, "quantized_moe_decode_gemv_gb300",
                                       "libmoe_gb300_checks.so")):
        pytest.fail("libmoe_gb300_checks.so is not built; run __graft_entry__.build()")
    env = dict(os.environ, MOE_CHECKS="1")
    env.pop("MOE_DEBUG_BAD_INDEX", None)
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])
    assert [c[2] for c in res["clean"]] == ["MOE_OK"] * 3, res
    (m1, st1, msg1, after1), (m2, st2, msg2, after2) = res["planted"]
    assert st1 == "MOE_ERR_INDEX" and "expert id" in msg1 and "outside [0, 16)" in msg1, res
    assert st2 == "MOE_ERR_INDEX" and "pair id" in msg2 and "outside [0, 2)" in msg2, res
    assert after1 == "MOE_OK" and after2 == "MOE_OK", res
