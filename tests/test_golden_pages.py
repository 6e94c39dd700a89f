"""Values the pages print (tests/golden/*.json, each with its source section)."""
import json
import os

import numpy as np

import oracle
from voxel_gemm_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_kernel_signature_fixture():
    g = json.load(open(os.path.join(GOLD, "masked_igemm_signature.json")))
    for logn, ci, co, V, _tf32 in g["key_examples"]:
        assert V == 27
        n = 1 << logn
        coords = synth.random_coords(logn, n, 1, 32, 32, 32)
        nbr, mask = oracle.nbrmap(coords, 1, 32, 32, 32)
        # neighbour table is uint32 [N, V]; the contraction runs over V * Ci
        assert nbr.dtype == np.dtype(g["arg_dtypes"]["neighbor"]) and nbr.shape == (n, V)
        rng = np.random.default_rng(0)
        f = rng.standard_normal((n, ci))
        W = rng.standard_normal((V, ci, co))
        out = oracle.fwd(nbr[:8], f, W, None)
        assert out.shape == (8, co)
        # one output = a single dot product of length V*Ci over the gathered rows
        gathered = np.concatenate([f[j] if j != oracle.NONE else np.zeros(ci) for j in nbr[0]])
        assert np.allclose(out[0], gathered @ W.reshape(V * ci, co), rtol=1e-12, atol=1e-12)
