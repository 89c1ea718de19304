"""The CTA-pair GEMM mode (tcgen05 cta_group::2, two SMs per unit; two weight
tiles per CTA where every segment has a multiple of four) is a tuning switch
read once per process, so its parity is checked by re-running the
packed-weight expert and layer parity tests in a child process with the
switch on for both expert passes -- including the full-size K2 prefill layer,
whose shared expert reads its token tiles through a tensor map in halves."""
import os
import subprocess
import sys

import pytest

from _gpu_common import need_gpu

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_pair_mode_parity_in_child_process():
    need_gpu()
    env = dict(os.environ, FGS_PAIR_GATE_UP="1", FGS_PAIR_DOWN="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
           os.path.join(HERE, "test_gpu_experts.py"), os.path.join(HERE, "test_gpu_layer.py"),
           "-k", "packed or bf16 or (full_size and k2_prefill)"]
    r = subprocess.run(cmd, env=env, cwd=os.path.dirname(HERE), capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
