"""The whole per-layer path with every fp32 GEMM on the FFMA kernels (GPTQ_FFMA_GEMM=1):
no tensor maps, so the factor runs without its look-ahead (panels wait for whole
trailing updates) and the lazy update takes the FFMA GEMM. The switch is read once per
process, so the check runs in a child process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from oracle import gptq_oracle as orc
from post_weight_quantization_gb300 import gptq as g
from synth import ActSpec, bf16_bits_to_f32, make_activations, make_weight

m, d, n = 160, 512, 4096
W = bf16_bits_to_f32(make_weight(m, d, 21))
X = bf16_bits_to_f32(make_activations(ActSpec("heavy_tail", n, d, seed=21))).astype(np.float64)
H = orc.hessian([X])
Hg = torch.from_numpy(H.astype(np.float32)).cuda()
U, _, info = g.gptq_factor(Hg, percdamp=0.01)
assert info == -1
Hd, _ = orc.damp(H.astype(np.float32).astype(np.float64), 0.01)
Uo = orc.hinv1(Hd)
rel = np.linalg.norm(U.cpu().numpy().astype(np.float64) - Uo) / np.linalg.norm(Uo)
assert rel < 50 * np.linalg.cond(Hd) * 2.0 ** -24, rel
U32 = Uo.astype(np.float32)
q = g.gptq_quantize_layer(torch.from_numpy(W).cuda(), torch.from_numpy(U32).cuda(), bits=4, group_size=128,
                          blocksize=128, sync=True)
codes = g.gptq_unpack_codes(q.qweight, m, d, 4).cpu().numpy().astype(np.int64)
res = orc.gptq_columns(W, U32, 4, 128, 128, dtype=np.float32)
mism = float(np.mean(codes != res["codes"]))
assert mism <= 0.005, mism
g.gptq_device_check()
print("ok", rel, mism)
"""


def test_path_through_ffma_gemms():
    env = dict(os.environ, GPTQ_FFMA_GEMM="1")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().startswith("ok"), r.stdout
