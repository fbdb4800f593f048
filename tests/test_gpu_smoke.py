"""The build/smoke entry point, run as part of the GPU suite."""

import pytest


@pytest.mark.gpu
def test_smoke_entry_point():
    import __graft_entry__ as g
    g.smoke()
