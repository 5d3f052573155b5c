"""The column loop's two kernel paths agree bit for bit: the outer-block kernel
(colmma_kernel, the K = 128 lazy updates on each SM's tensor core) and the per-block
kernels with the lazy updates as separate tensor-core GEMMs (GPTQ_COLUMN_KERNEL=chain)
form the same products with the same rounding ("GPTQ, Line by Line", the blocks of 128
columns and their lazy updates). Each path runs in a fresh process (the selection is
read once per process) on the same seeded W and the same Hessian, computed in float64
from the seeded tokens so that it does not depend on the order of the GPU's sums."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import hashlib, json, os, sys
import numpy as np, torch
sys.path.insert(0, ROOT); sys.path.insert(0, os.path.join(ROOT, "tests"))
from post_weight_quantization_gb300 import gptq as g
from synth import ActSpec, make_activations, make_weight
out = {}
for (m, d, n, bits, gs, ao, seed) in CASES:
    W = torch.from_numpy(make_weight(m, d, seed).view(np.int16)).cuda().view(torch.bfloat16)
    Xb = make_activations(ActSpec("heavy_tail", n, d, seed=seed + 1)).view(np.int16)
    Xd = torch.from_numpy(Xb).cuda().view(torch.bfloat16).double()
    H = (2.0 * (Xd.T @ Xd)).float().contiguous()
    U, perm, _ = g.gptq_factor(H, percdamp=0.01, act_order=ao)
    q = g.gptq_quantize_layer(W, U, perm, bits=bits, group_size=gs, blocksize=128)
    torch.cuda.synchronize()
    g.gptq_device_check()
    h = hashlib.sha256()
    for t in (q.qweight, q.scales, q.zeros, q.col_losses):
        h.update(t.cpu().numpy().tobytes())
    out[f"{m}x{d}-{bits}b-g{gs}-{int(ao)}"] = h.hexdigest()
print(json.dumps(out))
"""

# (m, d, tokens, bits, group, act-order, seed): ragged rows (300, 33, 1), a ragged last
# block (d = 1000), an outer block of one block (d = 1408 = 640 + 640 + 128), one row,
# per-channel and act-order, and the 4096-square layer
CASES = [(544, 1024, 8192, 4, 128, False, 3), (520, 1280, 4096, 2, 128, False, 4), (300, 1000, 4096, 3, -1, False, 5),
         (544, 1024, 8192, 4, 128, True, 6), (4096, 4096, 16384, 4, 128, False, 7), (1, 256, 512, 4, 128, False, 8),
         (33, 384, 1024, 8, 128, False, 9), (96, 1408, 2048, 4, 128, False, 10)]


def run_child(env_extra):
    env = dict(os.environ)
    env.pop("GPTQ_COLUMN_KERNEL", None)
    env.update(env_extra)
    code = f"ROOT = {ROOT!r}\nCASES = {CASES!r}\n" + CHILD
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    return json.loads(res.stdout.strip().splitlines()[-1])


def test_outer_block_kernel_matches_per_block_kernels():
    from post_weight_quantization_gb300 import build as b
    b.build()
    a = run_child({})
    c = run_child({"GPTQ_COLUMN_KERNEL": "chain"})
    assert a.keys() == c.keys()
    for k in a:
        assert a[k] == c[k], k
