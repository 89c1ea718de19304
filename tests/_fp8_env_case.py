"""Run in a child process by test_gpu_fp8.py: one small FP8 layer forward
under the library's tuning overrides given in the environment (read once per
process), printing a digest of the output bytes, so that two settings can be
compared bit for bit."""
import hashlib
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(1, os.path.dirname(HERE))

import torch  # noqa: E402

import synth  # noqa: E402
from test_gpu_fp8 import FP8_ENV_SHAPES, _forward  # noqa: E402


def main():
    shape = FP8_ENV_SHAPES[int(sys.argv[1])]
    g = synth.generate(shape, device="cuda")
    y, idx, w, counts = _forward(shape, g)
    torch.cuda.synchronize()
    h = hashlib.sha256(y.view(torch.int16).cpu().numpy().tobytes()).hexdigest()
    print("digest", h, int(torch.isfinite(y.float()).all()))


if __name__ == "__main__":
    main()
