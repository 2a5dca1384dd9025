"""Every dense GEMM kernel variant through the same oracle parity tests.

The library picks a kernel per problem: the 2SM kernel (tcgen05.mma.cta_group::2) with
256 x 384 tiles (BF16 output; two N = 192 MMAs sharing A), 256 x 256 tiles (the last,
partial wave of either as half tiles) or 256 x 192 tiles, or the one-SM kernel (128 x 256
or 128 x 128 tiles); grouped (MoE) GEMMs run on the 2SM kernel too (256-wide, 192-wide, or
384-wide for BF16 fprop / dgrad with N a multiple of 384), or on the one-SM kernel. The choice is read from the environment once per process, so each forced
variant runs the parity tests of test_gpu_gemm.py in a child process. The shapes there
cover ragged M, N and K, a CTA pair whose second M tile lies past M, and 192-wide tiles
starting 64 rows into a B scale tile.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
VARIANTS = {
    "2sm_256": {"MXFP8_GEMM_2SM": "1", "MXFP8_GEMM_BN": "256"},
    "2sm_256_whole_tiles": {"MXFP8_GEMM_2SM": "1", "MXFP8_GEMM_BN": "256",
                            "MXFP8_GEMM_HALF_TAIL": "0"},
    "2sm_192": {"MXFP8_GEMM_2SM": "1", "MXFP8_GEMM_BN": "192"},
    "2sm_384": {"MXFP8_GEMM_2SM": "1", "MXFP8_GEMM_BN": "384"},
    "2sm_384_whole_tiles": {"MXFP8_GEMM_2SM": "1", "MXFP8_GEMM_BN": "384",
                            "MXFP8_GEMM_HALF_TAIL": "0"},
    "1sm": {"MXFP8_GEMM_2SM": "0"},
}
SELECT = ("shapes_random_operands or extreme_scales or small_layer or layer_set_full_size "
          "or grouped_fprop_dgrad_wgrad_small or grouped_rows_bf16_384_wide_tiles "
          "or experts_full_size")


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_gemm_variant_parity(name):
    env = dict(os.environ)
    for key in ("MXFP8_GEMM_2SM", "MXFP8_GEMM_BN", "MXFP8_GEMM_HALF_TAIL", "MXFP8_GEMM_WIDE"):
        env.pop(key, None)
    env.update(VARIANTS[name])
    cmd = [sys.executable, "-m", "pytest", "tests/test_gpu_gemm.py", "-q", "-x", "-m", "gpu",
           "-k", SELECT, "-p", "no:cacheprovider"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, f"variant {name}:\n{r.stdout[-4000:]}\n{r.stderr[-2000:]}"
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1], r.stdout[-500:]
