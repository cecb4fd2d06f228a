"""Device-side failure detection without a GPU fault: a device wait that runs
out is reported as a status, and the CUDA context stays usable.

LCE_TEST_FORCE_TIMEOUT makes lce_forward's logits kernel issue no operand
loads, so the MMA issuer's bounded wait (2 s) runs out; the kernel records the
timeout bit, unwinds (drains, frees TMEM, meets its pair at the cluster
barrier) and returns. Nothing traps, faults or hangs."""
import numpy as np
import pytest

import oracle
from chunked_lm_head_linear_gb300 import inputs

pytestmark = pytest.mark.gpu


def _dev(N=300, d=128, V=1500, seed=41):
    import torch
    w = inputs.Workload("fault", N=N, d=d, V=V, sigma_w=0.05, ignore="random", ignore_frac=0.1, seed=seed)
    inp = inputs.make_inputs(w)
    H = torch.from_numpy(inp["H"].view(np.int16)).view(torch.bfloat16).cuda()
    W = torch.from_numpy(inp["W"].view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.from_numpy(inp["y"]).cuda()
    return inp, H, W, y


def test_forced_wait_timeout_is_reported_and_context_survives(cuda_lib):
    import torch
    inp, H, W, y = _dev()
    with pytest.raises(cuda_lib.LCEError) as e:
        cuda_lib.lce_forward(H, W, y, sync_check=True, reserved=cuda_lib.LCE_TEST_FORCE_TIMEOUT)
    assert e.value.code == cuda_lib.LCE_ERR_TIMEOUT
    # without sync_check the call returns at once; the bit is in the workspace
    ws = torch.empty(cuda_lib.workspace_size(cuda_lib.LCE_OP_FORWARD, *H.shape, W.shape[0]), dtype=torch.uint8,
                     device="cuda")
    cuda_lib.lce_forward(H, W, y, workspace=ws, reserved=cuda_lib.LCE_TEST_FORCE_TIMEOUT)
    assert cuda_lib.read_device_status(ws) & cuda_lib.LCE_DEVICE_TIMEOUT
    # the context is intact: a normal call on the same workspace is correct and clears the bit
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"], grads=False)
    loss, lse = cuda_lib.lce_forward(H, W, y, workspace=ws, sync_check=True)
    assert cuda_lib.read_device_status(ws) == 0
    assert abs(loss.item() - ref["loss"]) <= 1e-3 * ref["loss"]
    np.testing.assert_allclose(lse.cpu().numpy(), ref["lse"], rtol=1e-4)


def test_test_value_rejected_elsewhere(cuda_lib):
    _, H, W, y = _dev(N=64, d=64, V=300)
    for call in (lambda: cuda_lib.lce_fwd_bwd(H, W, y, reserved=cuda_lib.LCE_TEST_FORCE_TIMEOUT),
                 lambda: cuda_lib.lce_backward(H, W, y, y.float(), reserved=cuda_lib.LCE_TEST_FORCE_TIMEOUT)):
        with pytest.raises(cuda_lib.LCEError) as e:
            call()
        assert e.value.code == cuda_lib.LCE_ERR_INVALID_ARG
