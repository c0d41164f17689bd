"""H3_DEBUG_SYNC=1: every entry point that launches work waits for its stream
and returns the device status, so a kernel-reported error surfaces at the call
that caused it instead of at a later h3_sync_status.  The variable is read once
per process, so the calls run in a child process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import torch
import joint_audio_video_gb300 as h3
h3.load()
dev = "cuda"
# a bounded wait that nothing satisfies: the call itself reports the timeout
try:
    h3.h3_selftest_wait_timeout(2_000_000)
    print("timeout: no error")
except RuntimeError as e:
    print("timeout:", e)
# a modality id past n_mod: the modulate call itself reports the bad index
L, d = 4, 128
x = torch.randn(L, d, device=dev).to(torch.bfloat16)
z = torch.zeros(3, d, device=dev)
y = torch.empty_like(x)
bad = torch.tensor([0, 1, 7, 2], dtype=torch.uint8, device=dev)
try:
    h3.h3_adaln_modulate(x, bad, z, z, L, d, 3, 1e-6, y)
    print("bad index: no error")
except RuntimeError as e:
    print("bad index:", e)
# and a good call afterwards returns normally
h3.h3_adaln_modulate(x, torch.zeros(L, dtype=torch.uint8, device=dev), z, z, L, d, 3, 1e-6, y)
print("after:", h3.h3_sync_status())
"""


def test_debug_sync_reports_at_the_failing_call(h3):
    env = dict(os.environ, H3_DEBUG_SYNC="1")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = dict(l.split(":", 1) for l in r.stdout.strip().splitlines())
    assert "timeout" in lines["timeout"].lower() and "no error" not in lines["timeout"]
    assert "index" in lines["bad index"].lower() and "no error" not in lines["bad index"]
    assert lines["after"].strip() == "0"
