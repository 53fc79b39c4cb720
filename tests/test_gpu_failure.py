"""Failure detection without a GPU fault.

* A bounded device-side wait that runs out: the radix sort's decoupled
  look-back polls words that earlier tiles publish.  TOPK_OPT_SORT_WITHHOLD
  makes the first tile of each pass withhold its word (a flag that nothing
  sets), and TOPK_OPT_SORT_SPINS lowers the poll limit, so the tile after it
  gives up, every time.  A tile that gives up has summed only some earlier
  tiles, so its offsets are too small but never below its digit's base:
  every write stays inside the output (the order is wrong).
  topk_check_stream must then report TOPK_ERR_DEVICE_TIMEOUT, and the next
  sort, with both options cleared, must be right again.  The mbarrier waits
  on in-flight bulk copies are not shortened by any option.
* A host-side allocation failure (TOPK_OPT_FAULT_ALLOC, or the environment
  variable TOPK_FAULT_ALLOC=1): the call returns TOPK_ERR_NO_MEMORY and
  touches nothing; after the hook is cleared the same call succeeds.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tk():
    import topk_selection_gb300

    return topk_selection_gb300


def test_sort_lookback_gives_up_and_is_reported(tk):
    keys = synth.i32_uniform(50_000_017, 31).view(np.uint32)
    d = torch.from_numpy(keys.view(np.int32)).cuda()
    s = torch.cuda.Stream()
    tk.check_stream(s)  # start from a clean status word
    tk.set_option(tk.OPT_SORT_SPINS, 64)
    tk.set_option(tk.OPT_SORT_WITHHOLD, 1)
    try:
        with torch.cuda.stream(s):
            tk.sort_u32(d, stream=s)
        with pytest.raises(tk.TopKError) as err:
            tk.check_stream(s)
        assert err.value.status == 5  # TOPK_ERR_DEVICE_TIMEOUT
    finally:
        tk.set_option(tk.OPT_SORT_WITHHOLD, 0)
        tk.set_option(tk.OPT_SORT_SPINS, 0)
    with torch.cuda.stream(s):
        ko, _ = tk.sort_u32(d, stream=s)
    tk.check_stream(s)  # the word was cleared, and nothing gave up this time
    assert np.array_equal(ko.cpu().numpy().view(np.uint32), np.sort(keys))


def test_allocation_failure_is_a_status(tk):
    x = synth.i32_uniform(1_000_003, 32)
    d = torch.from_numpy(x).cuda()
    s = torch.cuda.Stream()  # a stream without a workspace yet
    out = torch.full((20,), 7, dtype=torch.int32, device="cuda")
    tk.set_option(tk.OPT_FAULT_ALLOC, 1)
    try:
        rc = tk.topk_i32_ptr(d.data_ptr(), d.numel(), 20, out.data_ptr(), s.cuda_stream)
        assert rc == 3  # TOPK_ERR_NO_MEMORY
    finally:
        tk.set_option(tk.OPT_FAULT_ALLOC, 0)
    torch.cuda.synchronize()
    assert torch.all(out == 7)  # nothing was written
    rc = tk.topk_i32_ptr(d.data_ptr(), d.numel(), 20, out.data_ptr(), s.cuda_stream)
    assert rc == 0
    s.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.topk_i32(x, 20))


def test_allocation_failure_from_the_environment():
    code = ("import torch, numpy as np, topk_selection_gb300 as tk\n"
            "x = torch.arange(100000, dtype=torch.int32, device='cuda')\n"
            "o = torch.empty(20, dtype=torch.int32, device='cuda')\n"
            "print(tk.topk_i32_ptr(x.data_ptr(), x.numel(), 20, o.data_ptr(), 0))\n")
    env = dict(os.environ, TOPK_FAULT_ALLOC="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip().splitlines()[-1] == "3"
