"""The entry point's smoke run (one linear layer forward and backward per scheme,
checked against the oracle) exercised with the GPU tests."""
import pytest

pytestmark = pytest.mark.gpu


def test_smoke():
    import __graft_entry__

    __graft_entry__.smoke()
