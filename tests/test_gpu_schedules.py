"""Every schedule and tile shape the GEMMs can take, through the same parity
checks: each setting runs tests/schedule_case.py in a child process (the library
reads these switches once per process).  GB300 only."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))

SETTINGS = [
    {"MLPBLK_TILE": "128"},           # single-CTA 128 x 128 tiles
    {"MLPBLK_TILE": "192"},           # single-CTA 128 x 192 tiles
    {"MLPBLK_TILE": "256"},           # single-CTA 128 x 256 tiles
    {"MLPBLK_TILE": "pair192"},       # CTA pairs, 256 x 192 (K-major B only; others fall back)
    {"MLPBLK_TILE": "pair"},          # CTA pairs, 256 x 256
    {"MLPBLK_STREAMK": "0"},          # whole tiles only
    {"MLPBLK_STREAMK": "2"},          # the split schedule wherever rounds are not whole
    {"MLPBLK_GROUP_M": "3"},          # another raster
    {"MLPBLK_MAX_SMS": "38"},         # a quarter of the SMs
    {"MLPBLK_SIDE_NORM": "0"},        # RMSNorm backward in its own kernel at every width
    {"MLPBLK_MN3D": "0"},             # MN-major operands box by box
    {"MLPBLK_NORM_ROWS2": "0"},       # RMSNorm backward one row per CTA iteration at every width
]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("setting", SETTINGS, ids=lambda s: ",".join(f"{k}={v}" for k, v in s.items()))
def test_schedule_parity(setting):
    env = dict(os.environ)
    env.update(setting)
    r = subprocess.run([sys.executable, os.path.join(HERE, "schedule_case.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, f"{setting}: {r.stdout[-2000:]}\n{r.stderr[-4000:]}"
