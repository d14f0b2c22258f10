"""Child process of tests/test_gpu_wait_timeout.py (run on its own: it loads a
test build of the library, not the library itself).

Runs one decode step through the test build, whose split-KV stage barriers
expect more bytes than are ever copied and whose bounded waits give up after
a short limit, then reports the device error word and whether the CUDA
context still works, as one JSON line.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_cache_42_gb300 import binding, build  # noqa: E402
from paged_kv_cache_42_gb300 import workloads as wl  # noqa: E402
from tests import gpu_util as gu  # noqa: E402


def main():
    build.LIB_PATH = sys.argv[1]
    build.build = lambda *a, **k: build.LIB_PATH
    binding.init()
    binding.get_device_error(clear=True)
    # head_dim 64: the CUDA-core split-KV kernel (the tensor-core one takes 128)
    w = wl.make_workload([200, 90, 700], [1, 1, 1], num_q_heads=4, num_kv_heads=2, head_dim=64,
                         seed=1301)
    b = gu.DeviceBatch(w)
    b.step()
    torch.cuda.synchronize()
    code, detail = binding.get_device_error(clear=True)
    # the context is still usable: a fresh allocation, a kernel and a copy back
    x = torch.arange(1000, device="cuda", dtype=torch.float32)
    usable = bool(float((x * 2).sum().item()) == 999000.0)
    print(json.dumps({"code": code, "detail": detail, "usable": usable}))


if __name__ == "__main__":
    main()
