"""The package's example (fsdp_sharded_optimizer_zero_gb300/example.py) runs as written on
the GPU, so the documented calls stay in step with the binding."""
import pytest

pytestmark = pytest.mark.gpu


def test_package_example_runs():
    import __graft_entry__ as g
    g.build()
    import torch
    from fsdp_sharded_optimizer_zero_gb300 import example
    master, param, Y = example.main()
    torch.cuda.synchronize()
    # the example's zero inputs give an exactly zero update and zero outputs
    assert torch.count_nonzero(master) == 0 and torch.count_nonzero(param.float()) == 0
    assert torch.count_nonzero(Y) == 0
