"""TRIMUL_LOG: one stderr line per tiled kernel launch, and nothing without it.

Each case runs a small forward (and a backward) in a child process, so that
the variable is read at create exactly as a user's process would read it.
The forward's logged launches must be the count the library reports for it
(trimul_kernels_per_forward).
"""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, torch
from co_folding_pair_gb300 import synthetic as S, trimul as T
w = S.custom(1, 136, 64, 64, seed=5, mask_kind="random_frac", mask_frac=0.2)
z, m, params = S.make_case(w, device="cuda")
h = T.trimul_create(params)
print("KPF", T.trimul_kernels_per_forward(h, 1, 136), flush=True)
sys.stderr.write("FWD-BEGIN\n"); sys.stderr.flush()
T.trimul_forward(h, z, m, "outgoing", flags=T.FLAG_CHECK)
sys.stderr.write("FWD-END\n"); sys.stderr.flush()
dout = torch.randn(z.shape, dtype=torch.float32, device="cuda").to(torch.bfloat16)
T.trimul_backward(h, z, m, dout, "incoming", flags=T.FLAG_CHECK)
torch.cuda.synchronize()
T.trimul_destroy(h)
"""


def run_child(log_value):
    env = dict(os.environ)
    env.pop("TRIMUL_LOG", None)
    if log_value is not None:
        env["TRIMUL_LOG"] = log_value
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout, r.stderr


def test_log_lines_match_the_launches():
    out, err = run_child("1")
    kpf = int(next(l.split()[1] for l in out.splitlines() if l.startswith("KPF")))
    lines = err.splitlines()
    assert any(l.startswith("trimul: create device") for l in lines), err[-2000:]
    fwd = lines[lines.index("FWD-BEGIN") + 1:lines.index("FWD-END")]
    fwd = [l for l in fwd if l.startswith("trimul: ")]
    kinds = [l.split()[1] for l in fwd]
    assert kinds[0] == "k1_inproj" and kinds[-1] == "k3_outproj", fwd
    assert set(kinds[1:-1]) == {"k2_triangle"}, fwd
    assert len(fwd) == kpf, (len(fwd), kpf, fwd)
    bwd = [l.split()[1] for l in lines[lines.index("FWD-END") + 1:] if l.startswith("trimul: ")]
    for k in ("k1_inproj", "k2_triangle", "k4_gemm", "k6_gate_grad"):
        assert k in bwd, (k, bwd)
    assert any("+ zh" in l for l in lines if l.startswith("trimul: k1_inproj")), "the recompute stores zh"


@pytest.mark.parametrize("value", [None, "0", ""])
def test_no_log_without_the_variable(value):
    _, err = run_child(value)
    assert not any(l.startswith("trimul: ") for l in err.splitlines()), err[-2000:]
