"""The C ABI from C: tests/c_abi_forward.c runs the whole Standard layer
(bf16, softmax top-2, M=64 K=256 N=128 E=8) through include/gbmoe.h alone,
with no Python in the process; its output is checked against the oracle."""
import re
import subprocess

import numpy as np
import pytest

import c_example
import oracle as orc
from gpu_common import TOL, assert_close_rel
from workloads import BF16

pytestmark = pytest.mark.gpu

M, K, N, E, TOPK = 64, 256, 128, 8, 2


def _bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_c_caller_runs_the_layer(tmp_path):
    exe = c_example.build(str(tmp_path))
    dumps = []
    for i in range(2):
        dump = tmp_path / f"run{i}.bin"
        r = subprocess.run([exe, str(dump)], capture_output=True, text=True, timeout=120)
        assert r.returncode == 0, r.stdout + r.stderr
        assert re.search(r"sum\|out\| = [0-9.]+", r.stdout), r.stdout
        dumps.append(dump.read_bytes())
    assert dumps[0] == dumps[1]  # separate processes, the same bits
    raw = dumps[0]
    sizes = [("x", np.uint16, (M, K)), ("logits", np.float32, (M, E)),
             ("w1", np.uint16, (E, 2 * N, K)), ("w2", np.uint16, (E, K, N)),
             ("out", np.uint16, (M, K))]
    a, off = {}, 0
    for name, dt, shape in sizes:
        n = int(np.prod(shape)) * np.dtype(dt).itemsize
        a[name] = np.frombuffer(raw[off:off + n], dt).reshape(shape)
        off += n
    assert off == len(raw)
    W = orc.Weights(orc.BF16, w1=a["w1"], w2=a["w2"])
    ref, _, _ = orc.moe_forward(a["x"], a["logits"], None, TOPK, orc.SOFTMAX, W)
    assert_close_rel(_bf16_to_f64(a["out"]), ref, TOL[BF16], "C caller vs oracle")
