"""The failure path on a GPU without a fault: a bounded wait that runs out reports TIMEOUT
through the device error word, once, and the context stays usable afterwards."""
import pytest
import torch

import fibattn_inputs as fi
import oracle
import static_fibonacci_offset_fibattn_b300 as fa
from gpu_common import TOL, f64, lib_schedule, max_abs, oracle_table, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    fa.poll_device_error()  # start clean
    fa.debug_wait_timeout(50)
    with pytest.raises(fa.FibAttnError) as e:
        fa.poll_device_error()
    assert e.value.status == fa.TIMEOUT
    fa.poll_device_error()  # the word was cleared
    # the context still runs the attention correctly
    sched = dict(kind="fixed", base="fib", alpha=(1, 1), n_layers=1)
    inp = fi.draw((1, 1, 2, 300, 64), seed=3, scale=0.5, dtype="bf16")
    dev = to_dev(inp)
    o, _ = fa.fwd(dev["q"], dev["k"], dev["v"], 16, lib_schedule(sched))
    torch.cuda.synchronize()
    fa.poll_device_error()
    ro, _ = oracle.fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), 16, oracle_table(sched, 0, 16, 300))
    assert max_abs(f64(o), ro) <= TOL["bf16"]
