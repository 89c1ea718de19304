"""Run in a child process by test_gpu_router.py: one router parity case under
the library's tuning overrides given in the environment (read once per
process), e.g. a K-part count that splits d / 64 unevenly."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(1, os.path.dirname(HERE))

import synth  # noqa: E402
from test_gpu_router import _check_router_from_x  # noqa: E402


def main():
    name, T = sys.argv[1], int(sys.argv[2])
    shape = synth.shape(name)
    g = synth.generate(shape, device="cuda", T=T, weights=False)
    _check_router_from_x(shape, g["x"], g["W_r"], g["bias"], tensor_cores=True)
    print("ok")


if __name__ == "__main__":
    main()
