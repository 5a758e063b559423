"""The GEMM kernel in each cluster size: single CTAs (CODA_CTA_PAIR=0), CTA
pairs only (CODA_CTA_QUAD=0), the per-GEMM policy CODA_CTA_QUAD=2 and split
launches (CODA_SPLIT=1: a two-pair kernel and a pair kernel share the GPU);
and the launch options turned off: programmatic
dependent launch (CODA_PDL=0), streaming epilogue stores for large
outputs (CODA_L2_HINTS=0), CTA pairs for GEMMs whose two-pair units fill
the last wave poorly (CODA_PAIR_WAVES=0), the L2 prefetch of the
epilogues' auxiliary rows (CODA_AUX_PREFETCH=0) and the shared-memory
staging of the QK-norm + RoPE backward map's rows (CODA_QK_TMA=0) and the
TMA ring that brings the plain epilogue's residual into shared memory
(CODA_EPI_RING=0), and the plain epilogue's chunk loops compiled per
feature set (CODA_EPI_LEAN=0 runs the general loop), and the RMSNorm-linear
backward's two GEMMs on half the grid each (CODA_RMS_SHARE=0 gives each the
whole grid), and the e4m3 row quantiser's shared-memory staging
(CODA_QROW_SMEM=0 runs a warp per row); and the defaults.  The
switches are read once per process, so each variant runs
cluster_variant_check.py (block forward/backward, FP8 linear, against the
fp64 oracle) in a fresh process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("env", [{"CODA_CTA_PAIR": "0"}, {"CODA_CTA_QUAD": "0"}, {"CODA_CTA_QUAD": "2"},
                                 {"CODA_SPLIT": "1"}, {"CODA_PDL": "0"}, {"CODA_L2_HINTS": "0"},
                                 {"CODA_PAIR_WAVES": "0"}, {"CODA_AUX_PREFETCH": "0"}, {"CODA_QK_TMA": "0"},
                                 {"CODA_EPI_RING": "0"}, {"CODA_EPI_LEAN": "0"}, {"CODA_RMS_SHARE": "0"},
                                 {"CODA_QROW_SMEM": "0"}, {}])
def test_cluster_variant(env):
    e = dict(os.environ)
    e.update(env)
    r = subprocess.run([sys.executable, os.path.join(HERE, "cluster_variant_check.py")], env=e,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), f"{env}:\n{r.stdout[-2000:]}\n{r.stderr[-4000:]}"
