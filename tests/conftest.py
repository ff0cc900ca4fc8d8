import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA device (B300, sm_103a) and the built library")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def v3_weights():
    """The V3 layer's weights (256 routed experts + shared, 22.5 GB of bf16)
    generated directly in device memory by the seeded input generator."""
    import torch
    from deepseekmoe_routing_expert_moe_b300 import inputs, ops
    cfg = inputs.CONFIGS["prefill_v3"]
    w1, w3, w2 = inputs.device_expert_weights(cfg, "cuda")
    ws1, ws3, ws2 = inputs.shared_weights(cfg, "cuda")
    wr = torch.from_numpy(inputs.router_weight(cfg)).cuda()
    torch.cuda.synchronize()
    return ops.Weights(wr, w1, w3, w2, ws1, ws3, ws2)
