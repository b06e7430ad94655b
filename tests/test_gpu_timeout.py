"""Bounded waits that run out, on the GPU, without faulting or hanging it.

Every pipeline wait in the tensor-core kernels is bounded; when one runs out the
kernel sets PIC_ERR_TIMEOUT in *err_flag, the other roles of the CTA give up at
their next wait (or at the barrier they share with a partner), copies in flight
are waited for, TMEM is freed, and the kernel returns.  To exercise that path
the library is built a second time with PIC_INJECT_WAIT_TIMEOUT: in that build
one role of each CTA of the link attention, the decode attention and the state
composition first waits on a barrier that nothing ever arrives on, with a 1 ms
bound.  A child process loads that build (PIC_LIBRARY), runs the three calls on
small bf16 workloads, reads the flag after each, and then runs a link step that
has no bounded waits (the fp32 worked example) to show that the context is
still usable; the parent process then runs a normal link step with the real
library."""

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import position_independent_kv_pic_gb300 as pic
from position_independent_kv_pic_gb300 import build as pic_build
from position_independent_kv_pic_gb300 import inputs
from position_independent_kv_pic_gb300.link import LinkBatch

from parity_util import TOL_MAX, TOL_MEAN, check_attention

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TEST_LIB = "libpic_waittest.so"
WAIT_NS = 1_000_000  # the injected wait's bound: 1 ms

CHILD = r'''
import json, os, sys
sys.path.insert(0, os.environ["PIC_ROOT"])
sys.path.insert(0, os.path.join(os.environ["PIC_ROOT"], "tests"))
import numpy as np
import torch
import position_independent_kv_pic_gb300 as pic
from position_independent_kv_pic_gb300 import inputs
from position_independent_kv_pic_gb300.link import LinkBatch
from position_independent_kv_pic_gb300.states import ComposeBatch
from parity_util import check_attention

assert os.path.basename(pic.library_path()) == os.environ["PIC_LIBRARY"]
res = {}
wl = inputs.custom([[130, 70, 45]], [21], [8], Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=1)
b = LinkBatch(wl)
b.run()
torch.cuda.synchronize()
res["attention"] = b.error()
b.setup_decode()
b.err.zero_()
b.run_decode()
torch.cuda.synchronize()
res["decode"] = b.error()
T, S, _ = inputs.linear_states(inputs.custom([[1] * 6], [1], [0], seed=3), H=4, d=128)
cb = ComposeBatch(T, S, [[0, 1, 2], [3, 4, 5, 0]])
cb.run()
torch.cuda.synchronize()
res["compose"] = cb.error()
# no bounded waits on this path (fp32 pools run the SIMT attention): it must still work
w = LinkBatch(inputs.worked_example())
w.run()
torch.cuda.synchronize()
res["after"] = w.error()
res["after_err"] = list(check_attention(w))
print("RESULT " + json.dumps(res))
'''


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    pic_build.build()
    pic.load()
    pic_build.build(extra_nvcc=[f"-DPIC_INJECT_WAIT_TIMEOUT={WAIT_NS}"], name=TEST_LIB)


def test_injected_wait_runs_out_cleanly():
    env = dict(os.environ, PIC_LIBRARY=TEST_LIB, PIC_ROOT=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT ")][-1]
    res = json.loads(line[len("RESULT "):])
    assert res["attention"] == pic.PIC_ERR_TIMEOUT, res
    assert res["decode"] == pic.PIC_ERR_TIMEOUT, res
    assert res["compose"] == pic.PIC_ERR_TIMEOUT, res
    assert res["after"] == 0, res
    emax, emean = res["after_err"]
    assert emax < 1e-5 and emean < 1e-6, res
    # and in this process, with the real library, a normal tensor-core link step
    b = LinkBatch(inputs.custom([[130, 70, 45]], [21], [8], Hq=32, Hkv=8, d=128, theta=5e5, dtype="bf16", seed=1))
    b.run()
    torch.cuda.synchronize()
    assert b.error() == 0
    emax, emean = check_attention(b)
    assert emax <= TOL_MAX and emean <= TOL_MEAN, (emax, emean)
