"""The grouped GEMM's shared-memory plan on the host (no GPU): for every tile
width, ring depth, A-tile count, chunks per slot and group size, the regions
the tensor copies and the 128-byte-swizzled MMA operands land in keep their
alignment -- ring slots, the B tile inside a slot and the dequantised A tiles
on 1024-byte boundaries (the swizzle atom), int4 code and scale/bias regions
on 128-byte boundaries (tensor-copy destinations) -- and each scale/bias copy
fits its region.  A misaligned tensor copy is a device fault, so this is
checked here, by compiling the plan function for the host with nvcc."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "quantized_moe_decode_gemv_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "moe_umma.cuh"
using namespace moe;
int main() {
  int bad = 0, n = 0;
  const int modes[2] = {UA_INT4, UA_DENSE};
  for (int mi = 0; mi < 2; ++mi)
    for (int gated = 0; gated < 2; ++gated)
      for (int nt = 16; nt <= 256; nt += 16)
        for (int st = 3; st <= UM_MAX_STAGES; ++st)
          for (int ab = 2; ab <= UM_MAX_ABUFS; ++ab)
            for (int sub = 1; sub <= 2; ++sub)
              for (int G : {32, 64, 128}) {
                const UmmaPlan p = umma_plan(modes[mi], gated != 0, nt, st, ab, sub, G);
                ++n;
                const bool ok = p.stage % 1024 == 0 && p.a_raw % 1024 == 0 && p.abuf % 1024 == 0 &&
                                p.b_tile % 1024 == 0 && p.code_bytes % 128 == 0 &&
                                (p.code_bytes + p.sb_bytes) % 128 == 0 && p.sb_box <= p.sb_bytes &&
                                p.tok % 16 == 0 && p.pref % 16 == 0 && p.total > p.pref;
                if (!ok && bad++ < 5)
                  std::printf("bad plan: mode %d gated %d n_tile %d stages %d abufs %d sub %d G %d\n",
                              modes[mi], gated, nt, st, ab, sub, G);
              }
  std::printf("%d plans, %d bad\n", n, bad);
  return bad != 0;
}
"""


def test_plan_regions_keep_their_alignment(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    src = tmp_path / "plan_check.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "plan_check"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17",
                    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                    str(src), "-o", str(exe)], check=True, capture_output=True, timeout=600)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout
    assert "0 bad" in r.stdout
