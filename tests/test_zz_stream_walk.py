"""The two-kernel step's walk (bs_stream_kernel + bs_merge_kernel) across the length
penalties and early-stopping modes.

The cluster kernel and the merge kernel each carry the walk, BeamHypotheses.add / is_done
and the pads; the cross of alpha and early_stopping elsewhere runs on shapes that take the
cluster kernel, so this one takes shapes that do not: 160 sentences of 4 beams (more
sentences than SMs) and W = 16 (2W candidates per row beyond one warp's merge).
"""

import pytest
import torch

from oracle import beam as ob
from tests import harness as hz

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from verify_bs_step_gb300 import _build
    _build.build()
    import verify_bs_step_gb300 as vbs
    return vbs.lib()


@pytest.mark.parametrize("es", [ob.ES_FALSE, ob.ES_TRUE, ob.ES_NEVER])
@pytest.mark.parametrize("lpk,alpha", [(ob.LP_GNMT, 0.6), (ob.LP_GNMT, 0.0), (ob.LP_POWER, 1.0)])
@pytest.mark.parametrize("kind,B,W,V,T", [
    ("sweep", 160, 4, 1024, 24),     # planted EOS hits; 4 to 25 of the 160 sentences finish
    ("tiny", 4, 16, 20, 40),         # V < 2W: EOS ranks high often, every sentence finishes but at alpha 1
])
def test_stream_path_walk(kind, B, W, V, T, es, lpk, alpha):
    case = hz.BeamCase(kind, B, W, V, T, torch.float32, eos=3, alpha=alpha, early_stopping=es, lp_kind=lpk,
                       seed=700 + B + W + es * 7 + int(alpha * 10))
    tr = hz.run_oracle(case)
    bs = hz.run_gpu_case(case, tr)
    hz.compare_finalize(case, tr, bs)
    hz.compare_finalize(case, tr, bs, n_return=W)
    bs.close()
