"""The round-trip smoke check of __graft_entry__ (one call of every operation
on cuda:0 against the oracle, and a training step through the autograd
functions) runs as a test too, so a change to a helper it shares with the
parity tests cannot break it unnoticed."""
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def test_smoke():
    import __graft_entry__
    __graft_entry__.smoke()
