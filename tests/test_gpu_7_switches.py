"""The stage graph's environment switches, each in a child process (both are
read once per process, at the first graph creation or launch).

ABG_TRACE=1: every graph launch synchronizes and prints one stderr line with
the launch count, the GPU milliseconds and the wall milliseconds.
ABG_PDL=0: launches are recorded without programmatic dependent launch, and a
batched call's launches after its first wait for the one before; the results
are the same bits as with it.
"""
from __future__ import annotations

import os
import re
import subprocess
import sys

import numpy as np
import pytest

import oracle
from affine_bit_group_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
abg = pytest.importorskip("affine_bit_group_gb300")
from affine_bit_group_gb300 import decode  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMALL = dict(seed=11, n_layers=2, hidden=1024, mlp=3072, head_rows=3000, q_rows=2048, kv_rows=256)

CHILD = """
import sys
sys.path.insert(0, {root!r})
import numpy as np, torch
import affine_bit_group_gb300 as abg
import oracle
from affine_bit_group_gb300 import decode, synth
model, h = synth.decode_model(**{small!r})
dm = decode.DeviceModel.upload(model)
g, out = decode.decode_token_graph(dm, torch.from_numpy(h).cuda(), fused={fused!r})
for _ in range({reps}):
    g.launch()
torch.cuda.synchronize()
got = out["logits"].cpu().numpy()
exp = oracle.decode_token(model, h)
print("LAUNCHES", g.launches)
print("EQUAL", int(np.array_equal(got.view(np.uint32), exp.view(np.uint32))))
print("HASH", oracle.hash32(got))
"""


def child(env_extra, fused, reps):
    # the switches a test does not set are off in the child, whatever the
    # parent's environment holds
    env = {k: v for k, v in os.environ.items() if k not in ("ABG_PDL", "ABG_TRACE")}
    env.update(env_extra)
    code = CHILD.format(root=ROOT, small=SMALL, fused=fused, reps=reps)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    vals = dict(line.split(None, 1) for line in r.stdout.splitlines() if line and line.split()[0].isupper())
    return vals, r.stderr


def in_process_hash(fused):
    model, h = synth.decode_model(**SMALL)
    dm = decode.DeviceModel.upload(model)
    g, out = decode.decode_token_graph(dm, torch.from_numpy(h).cuda(), fused=fused)
    g.launch()
    torch.cuda.synchronize()
    got = out["logits"].cpu().numpy()
    g.close()
    return oracle.hash32(got)


@pytest.mark.parametrize("fused", [False, True])
def test_pdl_off_gives_the_same_bits(fused):
    vals, _ = child({"ABG_PDL": "0"}, fused, reps=2)
    assert vals["EQUAL"].strip() == "1"
    assert int(vals["HASH"]) == in_process_hash(fused)


def test_trace_prints_one_line_per_launch():
    vals, err = child({"ABG_TRACE": "1"}, True, reps=3)
    assert vals["EQUAL"].strip() == "1"
    lines = [l for l in err.splitlines() if l.startswith("abg: stage graph")]
    assert len(lines) == 3, err[-2000:]
    n = int(vals["LAUNCHES"])
    pat = re.compile(r"abg: stage graph (\d+) launches, GPU ([0-9.]+) ms, wall ([0-9.]+) ms")
    for l in lines:
        m = pat.fullmatch(l.strip())
        assert m, l
        assert int(m.group(1)) == n
        gpu, wall = float(m.group(2)), float(m.group(3))
        assert 0.0 < gpu and 0.0 < wall and gpu <= wall * 1.5 + 0.05


def test_trace_off_prints_nothing():
    vals, err = child({}, True, reps=1)
    assert vals["EQUAL"].strip() == "1"
    assert "abg: stage graph" not in err


CHILD_MM = """
import sys
sys.path.insert(0, {root!r})
import numpy as np, torch
import affine_bit_group_gb300 as abg
import oracle
from affine_bit_group_gb300 import synth
m, _ = synth.mid()
rng = np.random.default_rng(17)
X = np.stack([synth.activations(rng, m.cols) for _ in range(5)])
XS = np.stack([oracle.gsum(x) for x in X])
w = torch.from_numpy(m.w.view(np.int32)).cuda()
Y = torch.empty(5 * m.rows, device="cuda")
for _ in range(2):
    abg.q4mm(w, torch.from_numpy(m.scale).cuda(), torch.from_numpy(m.bias).cuda(), torch.from_numpy(X).cuda(),
             torch.from_numpy(XS).cuda(), Y, cols=m.cols)
torch.cuda.synchronize()
got = Y.view(5, m.rows).cpu().numpy()
exp = oracle.q4mm(*m.arrays(), X, XS, m.cols)
print("EQUAL", int(np.array_equal(got.view(np.uint32), exp.view(np.uint32))))
"""


@pytest.mark.parametrize("pdl", ["0", "1"])
def test_batched_pdl_switch_gives_the_same_bits(pdl):
    """Five tokens (two pair launches and a single-token launch, the later ones
    started early unless ABG_PDL=0): every token bit-exact either way."""
    env = {k: v for k, v in os.environ.items() if k != "ABG_TRACE"}
    env["ABG_PDL"] = pdl
    r = subprocess.run([sys.executable, "-c", CHILD_MM.format(root=ROOT)], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "EQUAL 1" in r.stdout


CHILD_ATQ = """
import sys
sys.path.insert(0, {root!r})
import numpy as np, torch
import affine_bit_group_gb300 as abg
import oracle
from affine_bit_group_gb300 import synth
c = synth.atq_case(np.random.default_rng(31), 8, 2, 128, 700, 300)
d = {{k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in c.items() if k != "pos"}}
y = torch.empty(c["q"].size, device="cuda")
ys = torch.empty(c["q"].size // 64, device="cuda")
for _ in range(2):
    abg.atq(d["q"], d["gate"], d["k"], d["v"], d["qn_w"], d["kn_w"], d["cos"], d["sin"], d["Kc"], d["Vc"], y, ys,
            pos=c["pos"])
torch.cuda.synchronize()
ey, eys, eK, eV = oracle.atq(**c)
same = all(np.array_equal(a.view(np.uint32), b.view(np.uint32)) for a, b in
           ((y.cpu().numpy(), ey), (ys.cpu().numpy(), eys), (d["Kc"].cpu().numpy(), eK), (d["Vc"].cpu().numpy(), eV)))
print("EQUAL", int(same))
"""


@pytest.mark.parametrize("pdl", ["0", "1"])
def test_atq_pdl_switch_gives_the_same_bits(pdl):
    """The atq call's four launches (the last three started early unless
    ABG_PDL=0): every output bit-exact to the oracle either way."""
    env = {k: v for k, v in os.environ.items() if k != "ABG_TRACE"}
    env["ABG_PDL"] = pdl
    r = subprocess.run([sys.executable, "-c", CHILD_ATQ.format(root=ROOT)], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "EQUAL 1" in r.stdout


CHILD_GDN = """
import sys
sys.path.insert(0, {root!r})
import numpy as np, torch
import affine_bit_group_gb300 as abg
import oracle
from affine_bit_group_gb300 import synth
rng = np.random.default_rng(41)
c = synth.gdn_case(rng)
xs = [rng.standard_normal(c["x"].size).astype(np.float32) for _ in range(3)]
d = {{k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in c.items()}}
H, D = c["S"].shape[0], c["S"].shape[1]
ys = [torch.empty(H * D, device="cuda") for _ in xs]
yss = [torch.empty(H * D // 64, device="cuda") for _ in xs]
dx = [torch.from_numpy(x).cuda() for x in xs]
for t in range(3):   # three tokens back to back, the state carried, no sync between
    abg.gdn(dx[t], d["conv"], d["state"], d["a"], d["b"], d["z"], d["A_log"], d["dt_bias"], d["nw"], d["S"], ys[t],
            yss[t])
torch.cuda.synchronize()
S, st, same = c["S"], c["state"], True
for t in range(3):
    ey, eys, S, st = oracle.gdn(**dict(c, x=xs[t], S=S, state=st))
    same &= np.array_equal(ys[t].cpu().numpy().view(np.uint32), ey.view(np.uint32))
    same &= np.array_equal(yss[t].cpu().numpy().view(np.uint32), eys.view(np.uint32))
same &= np.array_equal(d["S"].cpu().numpy().view(np.uint32), S.view(np.uint32))
print("EQUAL", int(same))
"""


@pytest.mark.parametrize("pdl", ["0", "1"])
def test_gdn_pdl_switch_gives_the_same_bits(pdl):
    """Three gdn tokens on one state back to back (each launch scheduled early
    unless ABG_PDL=0, reading its inputs after the previous one finished):
    every output and the final state bit-exact to the oracle either way."""
    env = {k: v for k, v in os.environ.items() if k != "ABG_TRACE"}
    env["ABG_PDL"] = pdl
    r = subprocess.run([sys.executable, "-c", CHILD_GDN.format(root=ROOT)], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "EQUAL 1" in r.stdout
