"""The build's smoke pass (``__graft_entry__.smoke``) as a GPU test."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


@pytest.mark.gpu
def test_smoke():
    import __graft_entry__ as g
    g.smoke()
