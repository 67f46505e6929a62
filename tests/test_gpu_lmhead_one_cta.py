"""GPU: the LM-head GEMMs in their one-CTA form (the form a device without
co-schedulable CTA pairs runs), selected with SLP_LMHEAD_CTA_PAIRS=0 in a
child process: oracle parity on small cases and a wait bound that runs out
(tests/lmhead_one_cta_check.py).  The child's default workspace differs from
this process's, which runs the pairs."""

import os
import subprocess
import sys

import pytest

import vocab_selected_token_gb300 as slp
from tests.gpu_util import device

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_one_cta_form_in_a_child_process():
    device()
    pairs_ws = slp.slp_lmhead_workspace_size(8192, 151936, 2560)
    env = dict(os.environ, SLP_LMHEAD_CTA_PAIRS="0")
    r = subprocess.run([sys.executable, "-m", "tests.lmhead_one_cta_check"], cwd=ROOT, env=env,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:]
    assert "one-CTA form OK" in r.stdout
    child_ws = int([ln for ln in r.stdout.splitlines() if ln.startswith("workspace ")][0].split()[1])
    assert child_ws != pairs_ws  # the child really ran the other geometry
