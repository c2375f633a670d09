"""moe_layer_forward_static: the layer forward for callers that cannot
allocate device memory, with the scratch in a fixed region inside the
library.  It must give what moe_layer_forward gives with a caller workspace.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from routed_mixture_experts_router_gb300 import binding, synth
from gpu_util import TOL_F32, make_case, rel_l2_max

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    binding.load()


@pytest.mark.parametrize("name,flags", [("decode_t1", 0), ("decode_t64_zipf", binding.MOE_FLAG_DETERMINISTIC),
                                        ("decode_t64_zipf", 0)])
def test_static_scratch_matches_workspace_path(name, flags):
    case = make_case(synth.WORKLOADS[name])
    ref = binding.layer_forward(case.x, case.layer, flags=flags)
    torch.cuda.synchronize()
    r = ref.cpu().double().numpy()
    for _ in range(2):  # two calls in a row share (and reuse) the fixed region
        out = binding.layer_forward_static(case.x, case.layer, flags=flags)
        torch.cuda.synchronize()
        err = rel_l2_max(out.cpu().double().numpy(), r)
        assert err < TOL_F32, f"max rel L2 {err:.3e}"


def test_static_scratch_rejects_oversize_batch():
    wl = synth.WORKLOADS["decode_t1"]
    case = make_case(wl)
    T = 1024  # needs ~25 MB of scratch at this geometry, above the 8 MiB region
    x = torch.zeros(T, wl.d_model, device="cuda")
    with pytest.raises(binding.MoeError) as ei:
        binding.layer_forward_static(x, case.layer)
    assert ei.value.rc == binding.MOE_ERR_WORKSPACE
