"""The entry point's smoke check (one small forward + backward on cuda:0
against the fp64 oracle) stays in step with the library's conventions."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_entry_point_smoke():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__ as entry
    entry.smoke()
