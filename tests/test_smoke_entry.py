"""The entry point's smoke check runs as a GPU test too, so a break in it (or
in the oracle calls it makes) shows up in the suite, not only at the end."""
import pytest


@pytest.mark.gpu
def test_graft_entry_smoke():
    import __graft_entry__ as g
    g.smoke()
