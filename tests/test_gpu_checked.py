"""The checked build (libvbs_checked.so: the library compiled with VBS_CHECKED, device bounds
checks on every indexed access whose index comes from data) on small parity cases.

Each case compares the results with the fp64 oracle as the other GPU tests do, then asks
the library whether any check failed since the last case.  A memory checker is not
available on the GPU pool; these checks stand in for it on the small configurations.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import bpd as obpd
from oracle import kv as okv
from tests import harness as hz

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def checked_library():
    from verify_bs_step_gb300 import _build
    import verify_bs_step_gb300 as vbs
    _build.build()
    _build.build(checked=True)
    vbs.lib()
    old = vbs.use_library(vbs.load_checked())
    yield
    vbs.use_library(old)


def _no_check_failed():
    import verify_bs_step_gb300 as vbs
    checked, site, index = vbs.checked_record()
    assert checked, "the checked build is not the one loaded"
    assert site == -1, f"bounds check {site} failed at index {index}"


@pytest.mark.parametrize("kind,B,W,V,T,dtype,eos,ld_pad", [
    ("tiny", 3, 2, 6, 8, torch.float32, 5, 0),              # the tiny batched case (cluster kernel)
    ("tiny", 4, 16, 20, 30, torch.float32, 3, 0),           # W = 16: stream and merge kernels
    ("sweep", 7, 3, 777, 10, torch.float32, 3, 0),          # element path
    ("sweep", 2, 4, 4096, 10, torch.bfloat16, 3, 8),        # row stride ld > V
    ("sweep", 160, 4, 1024, 12, torch.float32, 3, 0),       # more sentences than SMs
])
def test_beam_step_checked(kind, B, W, V, T, dtype, eos, ld_pad):
    case = hz.BeamCase(kind, B, W, V, T, dtype, eos=eos, alpha=0.6, seed=B * 7 + W + V % 13, ld_pad=ld_pad)
    tr = hz.run_oracle(case)
    bs = hz.run_gpu_case(case, tr)
    hz.compare_finalize(case, tr, bs)
    hz.compare_finalize(case, tr, bs, n_return=W)
    bs.close()
    _no_check_failed()


def test_two_pass_and_shards_checked():
    case = hz.BeamCase("sweep", 6, 4, 3000, 8, torch.bfloat16, eos=3, alpha=0.6, seed=61)
    tr = hz.run_oracle(case)
    hz.run_gpu_case(case, tr, two_pass=True).close()
    hz.run_gpu_case(case, tr, shards=[7, 1500]).close()
    _no_check_failed()


def test_kv_checked():
    import verify_bs_step_gb300 as vbs
    g = torch.Generator().manual_seed(3)
    src = (torch.randn(2, 2, 6, 3, 20, 8, generator=g) * 4).to(torch.bfloat16)
    dst = (torch.randn(2, 2, 6, 3, 20, 8, generator=g) * 4).to(torch.bfloat16)
    bi = np.array([1, 1, 0, 5, -1, 2], dtype=np.int32)
    exp = okv.reorder_naive(src.float().numpy(), dst.float().numpy(), bi, 13)
    d = dst.cuda()
    vbs.kv_reorder(src.cuda(), d, torch.from_numpy(bi).cuda(), 13)
    assert vbs.lib().vbs_stateless_status(None) == 0
    np.testing.assert_array_equal(d.float().cpu().numpy(), exp)
    # the paged cache through a short decode, its logical view against the naive oracle
    from tests.test_gpu_kv import _paged_decode
    _paged_decode(2, 3, 2, 2, 8, 5, 12, torch.bfloat16, seed=9)
    _no_check_failed()


def test_kv_parent_outside_the_cache_is_refused():
    """A parent row that is not a row of the cache copies nothing and reports VBS_EINPUT (the
    guard is in every build; this runs it in the checked one)."""
    import verify_bs_step_gb300 as vbs
    src = torch.arange(1 * 2 * 4 * 1 * 6 * 4, dtype=torch.float32).view(1, 2, 4, 1, 6, 4)
    dst = torch.zeros_like(src)
    bi = torch.tensor([1, 4, 0, 2], dtype=torch.int32)            # 4 is not a row of a 4-row cache
    d = dst.cuda()
    vbs.kv_reorder(src.cuda(), d, bi.cuda(), 6)
    assert vbs.lib().vbs_stateless_status(None) == vbs.EINPUT
    out = d.cpu()
    assert torch.equal(out[:, :, 1], torch.zeros_like(out[:, :, 1]))
    assert torch.equal(out[:, :, 0], src[:, :, 1]) and torch.equal(out[:, :, 3], src[:, :, 2])
    _no_check_failed()


@pytest.mark.parametrize("B,k,V,dtype", [(37, 5, 1000, torch.bfloat16), (11, 3, 77, torch.bfloat16),
                                         (16, 8, 4096, torch.float32)])
def test_bpd_checked(B, k, V, dtype):
    import verify_bs_step_gb300 as vbs
    base, props, heads = synth.geometric_prefix_proposals(B, k, V, seed=B * k + V, step=0)
    logits = synth.planted_rows(heads, V, seed=B + k, salt=1, dtype=dtype)
    khat, nxt = vbs.bpd_verify(logits.cuda(), props.to(torch.int32).cuda())
    lg = logits.float().numpy()
    ekh, enx = obpd.verify(lg, props.numpy())
    np.testing.assert_array_equal(khat.cpu().numpy(), ekh)
    np.testing.assert_array_equal(nxt.cpu().numpy(), enx)
    _no_check_failed()
